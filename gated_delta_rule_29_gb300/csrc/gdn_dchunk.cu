// gdn_dchunk.cu -- the chunk-parallel gradient pass of gdn_bwd on the tensor cores (sm_103a).
//
// Method (cuDNN Linear Attention page, "Semantics worth knowing": every variant has a full
// backward).  In the chunked form of the forward (the chunk kernel's header), a 64-token chunk
// with raw key and query rows K, Q, entering state S and the factors of its WY record (beta,
// sx = beta 2^b rk, sq = scale rq 2^b, sd = 2^{b_C - b} rk, T = (I + A)^{-1}, P) computes
//   X = beta V - sx (.) (K S),  D = T X,  O = sq (.) (Q S) + P D,  S' = 2^{b_C} S + K^T (sd (.) D).
// Given dO and the gradient dS' of the state leaving the chunk (which the state-gradient pass
// stores for every chunk), reverse mode gives, for each chunk independently of the others:
//   dD = P^T dO + sd (.) (K dS'),   dX = T^T dD,   dV = beta (.) dX,
//   dA = -strict_tril(dX D^T),      dP = tril(dO D^T),
//   dk~ = (-sx (.) dX) S^T + (sd (.) D) dS'^T + rk (.) [(M + M^T)(rk (.) K) + H^T (rq (.) Q)],
//   dq~ = (sq (.) dO) S^T + rq (.) [H (rk (.) K)],
//   M_ij = dA_ij beta_i 2^{b_i - b_j},  H_ij = dP_ij scale 2^{b_i - b_j},
// where dk~ = rk dk_hat is the gradient of the normalised row times its inverse norm, so that
// the L2-norm backward is dk = dk~ - rk^2 (k . dk~) k (and dq alike).  The per-token sums give
//   dbeta_i = sum_v dX (V - 2^{b_i} rk_i (K S)) + sum_j dA_ij rk_i rk_j (k_i . k_j) 2^{b_i - b_j},
//   db_i    = -sx_i sum_v dX (K S) + sq_i sum_v dO (Q S) + (row i - column i of dA (.) A)
//             + (row i - column i of dP (.) P) - w_i  [+ 2^{b_C} <dS', S> + sum_j w_j at the
//             chunk's last token],  w_j = sd_j sum_v (K dS')_jv D_jv,
// every decay factor differentiated with respect to its natural-log exponent, and the gate
// gradient dg_j = sum_{i >= j} db_i within the chunk.
//
// Mapping: one persistent CTA of 512 threads per SM takes (chunk, head) items in turn.  Every
// product is a tcgen05.mma (kind::f16, fp32 accumulation in TMEM, M = 128) from 128-byte
// swizzled shared-memory tiles; fp32 operands that reach dbeta, dg or dv are split into bf16 hi
// and lo parts, those that only reach the bf16 dk and dq are rounded once.  The accumulators
// take three orientations: value columns on the TMEM lanes for the V-wide products (as in the
// forward's state pass), tokens on the lanes for the 64 x 64 ones (dA, dP and the G product),
// key columns on the lanes for dk and dq.  Warps w, w + 4, w + 8 and w + 12 share a lane
// quadrant and split the columns into four groups.  Sums over the lanes are reduce-scatters by shuffles (a warp's 32 lanes hand each
// lane one column's sum), added over the four quadrants in a fixed order.  Every wait is bounded.
#include <cuda_bf16.h>

#include "../../include/liblinattn.h"
#include "gdn_kernel.h"
#include "ptx.cuh"
#include "gdn_device.cuh"

namespace la {
namespace {

constexpr int kDT = 512;  // threads
constexpr int kIo = 64;   // the thread that issues the copies (not in the gate-scan warps; thread 0 issues the products)
constexpr int kMmaLast = 96;  // the issuer of the last products (its warp has no token-row epilogue after them)
constexpr float kLog2eD = 1.4426950408889634f;

// Shared memory (byte offsets from the 1024-aligned base).  Phase by phase a region is reused
// once the products reading it have completed:
//   KQ     [K; Q] tile [region 0..1 (key columns)][128 rows][128 B]             whole item
//   ST     S^T hi [region 0..1 (key columns)][128 rows v][128 B]                 until dk~ += S W,
//          then the first half of the next item's S (fp32)
//   STLO   S^T lo -> X^T hi, lo -> D^T hi, lo
//   DST    dS'^T hi                                                              until acc2
//   DSTLO  dS'^T lo -> dD^T hi, lo -> [dX lo | dX hi | (TLO) dO^T] -> [N ; Hs] bf16 and a zero tile
//   TLO    T lo, P lo [64 rows][128 B] each -> dO^T (the MN-major A's upper half)
//   TB, PB T hi, P hi [64 rows][128 B] -> W region 0
//   DO     dO tile -> W region 1
// S arrives as fp32 [K][V] in ST..STLO (bulk copy, prefetched during the previous item) and is
// split in place; dS' likewise into DST..DSTLO.  V is read from global memory into registers,
// one value column per thread, when an item starts.  At the end of an item the output tiles are
// staged for TMA stores: dq in TLO..PLO, dk in TB..PB, dv in DO.
constexpr uint32_t D_KQ = 0;
constexpr uint32_t D_ST = 32768;
constexpr uint32_t D_STLO = 65536;
constexpr uint32_t D_DST = 98304;
constexpr uint32_t D_DSTLO = 131072;
constexpr uint32_t D_TLO = 163840;
constexpr uint32_t D_PLO = 172032;
constexpr uint32_t D_TB = 180224;
constexpr uint32_t D_PB = 188416;
constexpr uint32_t D_DO = 196608;
constexpr uint32_t D_SC = 212992;

// TMEM columns (fp32, 128 lanes): value-column accumulators first, then (their regions consumed)
// the token- and key-column ones; G stays from the first phase to the dA / dP phase.
constexpr uint32_t T_X1 = 0;     // [(K S)^T | (Q S)^T]
constexpr uint32_t T_X2 = 128;   // (K dS')^T
constexpr uint32_t T_DT = 192;   // D^T
constexpr uint32_t T_ET = 256;   // (P^T dO)^T
constexpr uint32_t T_DY = 320;   // dX^T
constexpr uint32_t T_G = 384;    // G = [K; Q] [K; Q]^T (token rows)
constexpr uint32_t T_DKQ = 0;    // [dk~ ; dq~] (token rows: dk~ 0-63, dq~ 64-127), 128 columns
constexpr uint32_t T_DAP = 128;  // [dX D^T ; dO D^T] (token rows)
constexpr uint32_t T_DAP2 = 192; // dX_lo D_hi^T (rows 0-63)
constexpr uint32_t T_ACC2 = 384; // D dS'^T (token rows 0-63; after G is read)
constexpr uint32_t T_COLS = 512;

struct __align__(16) DcScalars {
    float bet[64], sx[64], sq[64], sd[64];  // the WY record's factors (one bulk copy)
    float bw[64];                           // per-warp inclusive scans of g * log2(e)
    float b[64];                            // chunk-local inclusive cumsum of g * log2(e)
    float rk[64], rq[64];                   // inverse row norms (0 past the sequence end)
    float gr[64];                           // 2^{b_i} rk_i
    float gt[64];                           // the gates after the input transform (natural log)
    float psb[4][64], psg[4][64], pso[4][64], pw[4][64];  // per lane-quadrant sums over values
    float rowA[4][64], rowP[4][64], sbA[4][64];           // per column-group row sums
    float colA[2][64], colP[2][64];                       // per row-quadrant column sums
    float pdot[4][128];                                   // norm backward: partial k . dk~, q . dq~
    float db[64];
    float gp[4];
    float red[16];
    uint64_t bar_in, bar_pre, bar_mma, bar_mma2;
    uint64_t bar_pre0;  // the first half of S's fp32 staging, requested early
    uint32_t tmem_base;
    int32_t status0;
};
constexpr uint32_t D_SMEM = D_SC + static_cast<uint32_t>(sizeof(DcScalars)) + 1024;
static_assert(D_SMEM <= 232448, "gradient chunk pass: shared memory exceeds the per-CTA limit");

// Reduce-scatter over the warp: lane l returns the sum over the 32 lanes of element l of x
// (x is clobbered).  31 shuffles, fixed order.
__device__ __forceinline__ float scatter_sum32(float (&x)[32], int lane) {
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int e = 0; e < s; ++e) {
            const float send = up ? x[e] : x[e + s];
            const float keep = up ? x[e + s] : x[e];
            x[e] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
    return x[0];
}
// The same for 16 elements: lane l returns the sum over the 32 lanes of element l & 15
// (reduce-scatter within each half-warp, then the two halves added; 16 shuffles).
__device__ __forceinline__ float scatter_sum16(float (&x)[16], int lane) {
#pragma unroll
    for (int s = 8; s >= 1; s >>= 1) {
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int e = 0; e < s; ++e) {
            const float send = up ? x[e] : x[e + s];
            const float keep = up ? x[e + s] : x[e];
            x[e] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
    return x[0] + __shfl_xor_sync(0xffffffffu, x[0], 16);
}

// Column `col` (a value or key index) of a bf16 tile [region 0..1][rows][128 B] with regions
// `region_bytes` apart: element of row i.
__device__ __forceinline__ float tile_col(const uint8_t* tile, uint32_t region_bytes, int col, int i) {
    const uint8_t* p = tile + (col >> 6) * region_bytes + (col & 7) * 2;
    return bf16_bits_to_f(*reinterpret_cast<const uint16_t*>(p + sw128_off(static_cast<uint32_t>(i),
                                                                          static_cast<uint32_t>((col & 63) >> 3))));
}

// K-step offsets (descriptor units of 16 bytes) of the 16-wide slices along K: K-major operands
// with K = 128 over two 64-column regions 16 KB apart, K-major with K = 64, MN-major (16 rows).
__device__ __forceinline__ uint64_t koff128(int kk) { return static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4); }
__device__ __forceinline__ uint64_t koff64(int kk) { return static_cast<uint64_t>((kk * 32) >> 4); }
__device__ __forceinline__ uint64_t moff(int kk) { return static_cast<uint64_t>((kk * 2048) >> 4); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&x)[32]) {
    tmem_ld16(taddr, *reinterpret_cast<float(*)[16]>(&x[0]));
    tmem_ld16(taddr + 16, *reinterpret_cast<float(*)[16]>(&x[16]));
}
// 32 lanes x 32 bit, 8 consecutive columns.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&r)[8]) {
    uint32_t u[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 8; ++i) r[i] = __uint_as_float(u[i]);
}
// Reduce-scatter of 8 elements over the warp: lane l returns the sum over the 32 lanes of element
// l & 7 (9 shuffles).
__device__ __forceinline__ float scatter_sum8(float (&x)[8], int lane) {
#pragma unroll
    for (int s = 4; s >= 1; s >>= 1) {
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int e = 0; e < s; ++e) {
            const float send = up ? x[e] : x[e + s];
            const float keep = up ? x[e + s] : x[e];
            x[e] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
    float v = x[0] + __shfl_xor_sync(0xffffffffu, x[0], 8);
    return v + __shfl_xor_sync(0xffffffffu, v, 16);
}
// A bounded wait on an mbarrier phase in a compact loop (this kernel's code is large enough that
// an unrolled spin would crowd the instruction cache); false after budget_ns.
__device__ __noinline__ bool wait_phase(uint64_t* bar, uint32_t parity, uint64_t budget_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
#pragma unroll 1
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > budget_ns) return false;
    }
}

__global__ void __launch_bounds__(kDT, 1)
    gdn_dchunk_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap domap, const __grid_constant__ CUtensorMap wymap,
                      const __grid_constant__ CUtensorMap dkmap, const __grid_constant__ CUtensorMap dqmap,
                      const __grid_constant__ CUtensorMap dvmap, const ChunkArgs a, const BwdArgs bw) {
    constexpr int KD = 128;  // key and value width of this pass
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    DcScalars& sc = *reinterpret_cast<DcScalars*>(sm + D_SC);
    uint8_t* KQ = sm + D_KQ;
    uint8_t* ST = sm + D_ST;
    uint8_t* STLO = sm + D_STLO;
    uint8_t* DST = sm + D_DST;
    uint8_t* DSTLO = sm + D_DSTLO;
    uint8_t* TLO = sm + D_TLO;
    uint8_t* PLO = sm + D_PLO;
    uint8_t* TB = sm + D_TB;
    uint8_t* PB = sm + D_PB;
    uint8_t* DO = sm + D_DO;
    uint8_t* NH = sm + D_DSTLO;  // [N ; Hs] bf16 [128 rows][128 B], then an 8 KB zero tile
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int q4 = (tid >> 5) & 3;  // TMEM lane quadrant of this warp
    const int cg = tid >> 7;        // column group (16 of 64, or 32 of 128 columns)
    const int r = tid & 127;        // TMEM lane
    const int HO = a.HV;

    if (tid == 0) sc.status0 = *reinterpret_cast<volatile int32_t*>(&a.hdr->status);
    __syncthreads();
    if (sc.status0 != LA_OK) return;
    if (tid < 32) {
        tmem_alloc(&sc.tmem_base, T_COLS);
        tmem_relinquish();
    }
    if (tid == 0) {
        mbar_init(&sc.bar_in, 1);
        mbar_init(&sc.bar_pre, 1);
        mbar_init(&sc.bar_pre0, 1);
        mbar_init(&sc.bar_mma, 1);
        mbar_init(&sc.bar_mma2, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sc.tmem_base;
    const uint32_t trow = tmem + (static_cast<uint32_t>(32 * q4) << 16);

    // operand descriptors (an operand at byte offset off from a buffer uses base + (off >> 4))
    const uint64_t d_kq = sdesc_sw128(smem_u32(KQ), 16, 1024);            // [K; Q] rows, K-major
    const uint64_t d_kq_mn = sdesc_sw128(smem_u32(KQ), 16384, 1024);      // [K; Q]^T: key columns MN-major
    const uint64_t d_st = sdesc_sw128(smem_u32(ST), 16, 1024);            // S^T hi, K-major
    const uint64_t d_stlo = sdesc_sw128(smem_u32(STLO), 16, 1024);        // S^T lo
    const uint64_t d_s_mn = sdesc_sw128(smem_u32(ST), 16384, 1024);       // S hi: key rows MN-major
    const uint64_t d_dst = sdesc_sw128(smem_u32(DST), 16, 1024);          // dS'^T hi, K-major
    const uint64_t d_dstlo = sdesc_sw128(smem_u32(DSTLO), 16, 1024);      // dS'^T lo
    const uint64_t d_ds_mn = sdesc_sw128(smem_u32(DST), 16384, 1024);     // dS' hi: key rows MN-major
    const uint64_t d_xt = sdesc_sw128(smem_u32(STLO), 16, 1024);          // X^T hi (lo 16 KB on)
    const uint64_t d_tb = sdesc_sw128(smem_u32(TB), 16, 1024);            // T hi, K-major
    const uint64_t d_t_mn = sdesc_sw128(smem_u32(TB), 8192, 1024);        // T hi read MN-major
    const uint64_t d_tlo = sdesc_sw128(smem_u32(TLO), 16, 1024);          // T lo
    const uint64_t d_tlo_mn = sdesc_sw128(smem_u32(TLO), 8192, 1024);
    const uint64_t d_p_mn = sdesc_sw128(smem_u32(PB), 8192, 1024);        // P hi read MN-major
    const uint64_t d_plo_mn = sdesc_sw128(smem_u32(PLO), 8192, 1024);     // P lo
    const uint64_t d_do_mn = sdesc_sw128(smem_u32(DO), 8192, 1024);       // dO^T: value columns MN-major
    const uint64_t d_dd = sdesc_sw128(smem_u32(DSTLO), 16, 1024);         // dD^T hi (lo 16 KB on)
    const uint64_t d_dt_mn = sdesc_sw128(smem_u32(STLO), 16384, 1024);    // D^T hi as MN-major B (lo 16 KB on)
    const uint64_t d_ax_mn = sdesc_sw128(smem_u32(DSTLO + 16384), 16384, 1024);  // [dX hi ; dO (TLO)] MN-major
    const uint64_t d_axlo_mn = sdesc_sw128(smem_u32(DSTLO), 16384, 1024);        // [dX lo ; dX hi]
    const uint64_t d_w_mn = sdesc_sw128(smem_u32(TB), 16384, 1024);       // W = [-sx dX | sq dO]^T
    const uint64_t d_nh = sdesc_sw128(smem_u32(NH), 16, 1024);            // [N ; Hs], K-major (rows i)
    const uint64_t d_nt_mn = sdesc_sw128(smem_u32(NH), 16384, 1024);      // [N^T ; 0]: N read MN-major
    const uint64_t d_ht_mn = sdesc_sw128(smem_u32(NH + 8192), 8192, 1024);  // [Hs^T ; 0]
    const uint64_t budget = a.wait_budget_ns;
    // K and Q, dO, T hi (TMA), T lo, the factors (bulk); then S (fp32) and dS' (bulk)
    const uint32_t in_bytes = 2u * 16384u + 2u * 8192u + 2u * static_cast<uint32_t>(kWyTileBytes) +
                              static_cast<uint32_t>(kWyFactorBytes);
    constexpr uint32_t kPreBytes = 2u * 65536u;

    const int64_t total_items = a.chunk_off[a.N] * HO;
    uint32_t ph_in = 0, ph_pre = 0, ph_pre0 = 0, ph_mma = 0, ph_mma2 = 0;
    bool pend_in = false, pend_pre = false, pend_pre0 = false, pend_mma = false, pend_mma2 = false, failed = false;
    bool prefetched = false;  // this item's S and dS' were requested during the previous item
    // S (fp32, into ST..STLO) and dS' (into DST..DSTLO) of an item: S's first half (keys 0-63,
    // into ST) on bar_pre0, the rest on bar_pre.  ST is free once dk~ += W^T S^T has completed, so
    // the first half of the next item's S is requested then, the rest after the last products.
    // One thread.
    auto load_state_half = [&](int64_t it) {
        mbar_arrive_expect_tx(&sc.bar_pre0, 32768u);
        bulk_load(ST, bw.ckpt + it * static_cast<int64_t>(KD * KD), 32768u, &sc.bar_pre0);
    };
    auto load_states_rest = [&](int64_t it) {
        mbar_arrive_expect_tx(&sc.bar_pre, kPreBytes - 32768u);
        bulk_load(ST + 32768, bw.ckpt + it * static_cast<int64_t>(KD * KD) + KD * KD / 2, 32768u, &sc.bar_pre);
        bulk_load(DST, a.ds_chunks + it * 65536, 65536u, &sc.bar_pre);
    };
    auto load_states = [&](int64_t it) {
        load_state_half(it);
        load_states_rest(it);
    };
    // waits on the product barrier (every thread), folding the outcome into ok
    auto wait_mma = [&](bool& ok) {
        const bool okm = wait_phase(&sc.bar_mma, ph_mma, budget);
        if (okm) {
            ph_mma ^= 1u;
            pend_mma = false;
        }
        ok = ok && okm;
        tc_fence_after();
    };

    // an item's first token and length, and (threads 0-63) its token's gate after the transform;
    // read one item ahead, so that these dependent global loads stay off the item's path
    int64_t nt0 = 0;
    int nn = 0;
    float ngt = 0.f;
    uint16_t nv[16];  // V of value column r, tokens 16 cg .. (bf16 bits)
    auto item_meta = [&](int64_t it) {
        const int64_t chunk_ = it / HO;
        const int h_ = static_cast<int>(it % HO);
        const int seq_ = a.chunk_seq[chunk_];
        const int64_t c_ = chunk_ - a.chunk_off[seq_];
        const int64_t ts_ = cu_get(a.cu, a.cu64, seq_);
        const int64_t L_ = cu_get(a.cu, a.cu64, seq_ + 1) - ts_;
        nt0 = ts_ + c_ * kChunk;
        nn = static_cast<int>(L_ - c_ * kChunk < kChunk ? L_ - c_ * kChunk : kChunk);
        float gA_ = 0.f, gdt_ = 0.f;
        if (a.gate_mode == LA_GATE_SOFTPLUS) {
            gA_ = -expf(a.a_log[h_]);
            gdt_ = a.dt_bias[h_];
        }
        ngt = (tid < 64 && tid < nn) ? gate_at(a, nt0 + tid, h_, gA_, gdt_) : 0.f;
        const uint16_t* vp = bw.v + h_ * bw.v_sh + r;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const int i = 16 * cg + e;
            nv[e] = i < nn ? vp[(nt0 + i) * bw.v_st] : uint16_t(0);
        }
    };
    if (static_cast<int64_t>(blockIdx.x) < total_items) item_meta(blockIdx.x);

    for (int64_t item = blockIdx.x; item < total_items; item += gridDim.x) {
        const int64_t chunk = item / HO;
        const int h = static_cast<int>(item % HO);
        const int hk = h / a.group;
        const int64_t t0 = nt0;
        const int n = nn;
        const float gt_mine = ngt;
        float gAh = 0.f, gdt = 0.f;
        if (a.gate_mode == LA_GATE_SOFTPLUS) {
            gAh = -expf(a.a_log[h]);
            gdt = a.dt_bias[h];
        }

        // ---- P0: tiles, T, factors and dS' by TMA / bulk copy; S^T hi + lo from the fp32 state
        // the K/Q tile and the factors first (their buffers are no output's staging), then, once the
        // previous item's output tiles have left their staging buffers, dO, T and T's residual
        if (tid == kIo && !a.test_skip_tile_load) {  // (the failure-path test hook: no tile loads)
            mbar_arrive_expect_tx(&sc.bar_in, in_bytes);
#pragma unroll
            for (int rg = 0; rg < 2; ++rg) {
                tma_load_3d(KQ + rg * 16384, &kmap, &sc.bar_in, rg * 64, hk, static_cast<int>(t0));
                tma_load_3d(KQ + rg * 16384 + 8192, &qmap, &sc.bar_in, rg * 64, hk, static_cast<int>(t0));
            }
            bulk_load(sc.bet, a.wy + item * static_cast<int64_t>(kWyRecordBytes) + 2 * kWyTileBytes,
                      static_cast<uint32_t>(kWyFactorBytes), &sc.bar_in);
        }
        if (tid == kIo) {
            if (!prefetched) load_states(item);
            bulk_wait_read_all();  // the previous item's output tiles have left their staging buffers
        }
        if (tid == kIo && !a.test_skip_tile_load) {
#pragma unroll
            for (int rg = 0; rg < 2; ++rg)
                tma_load_3d(DO + rg * 8192, &domap, &sc.bar_in, rg * 64, h, static_cast<int>(t0));
            tma_load_3d(TB, &wymap, &sc.bar_in, 0, static_cast<int>(item), 0);
            bulk_load(TLO, a.wy_tlo + item * static_cast<int64_t>(kWyTileBytes), static_cast<uint32_t>(kWyTileBytes),
                      &sc.bar_in);
        }
        pend_in = !a.test_skip_tile_load;
        pend_pre = true;
        pend_pre0 = true;
        // V: this thread's value column r, tokens 16 cg .. (read one item ahead; for X and the dbeta sums)
        float vv[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) vv[e] = bf16_bits_to_f(nv[e]);
        if (tid < 64) {
            // gates: per-warp inclusive scans of g * log2(e) (rows past the end carry 0)
            const float gt = gt_mine;
            float x = gt * kLog2eD;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, x, off);
                if (lane >= off) x += y;
            }
            sc.gt[tid] = gt;
            sc.bw[tid] = x;
        }
        // this thread: value column r, key columns 32 cg .. 32 cg + 31 (region cg / 2, chunks 4 (cg % 2) ..)
        float s32[32];
        const uint32_t sreg = static_cast<uint32_t>(cg >> 1) * 16384u;
        const uint32_t sch = static_cast<uint32_t>(cg & 1) * 4u;
        bool ok = wait_phase(&sc.bar_pre0, ph_pre0, budget);
        if (ok) {
            ph_pre0 ^= 1u;
            pend_pre0 = false;
        }
        {
            const bool okp = wait_phase(&sc.bar_pre, ph_pre, budget);
            if (okp) {
                ph_pre ^= 1u;
                pend_pre = false;
            }
            ok = ok && okp;
        }
        {
            const float* Sf = reinterpret_cast<const float*>(ST) + (32 * cg) * KD + r;  // S[a][v], fp32 staging
#pragma unroll
            for (int e = 0; e < 32; ++e) s32[e] = ok ? Sf[e * KD] : 0.f;
        }
        __syncthreads();  // the fp32 staging is read: S^T hi + lo take its place
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
            const uint32_t off = sreg + sw128_off(r, sch + c4);
            store8_split(ST + off, STLO + off, &s32[8 * c4]);
        }
        {
            const bool oki = wait_phase(&sc.bar_in, ph_in, budget);
            if (oki) {
                ph_in ^= 1u;
                pend_in = false;
            }
            ok = ok && oki;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(!ok)) { failed = true; break; }

        // ---- P1: (K S)^T, (Q S)^T (S hi + lo), (K dS')^T (dS' hi + lo), G = [K; Q][K; Q]^T
        if (tid == 0) {
            tc_fence_after();
            const uint32_t i128 = idesc_bf16_f32(128, 128, false, false);
            const uint32_t i64 = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) umma_bf16(tmem + T_X1, d_st + koff128(kk), d_kq + koff128(kk), i128, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) umma_bf16(tmem + T_X1, d_stlo + koff128(kk), d_kq + koff128(kk), i128, 1u);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) umma_bf16(tmem + T_X2, d_dst + koff128(kk), d_kq + koff128(kk), i64, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) umma_bf16(tmem + T_X2, d_dstlo + koff128(kk), d_kq + koff128(kk), i64, 1u);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) umma_bf16(tmem + T_G, d_kq + koff128(kk), d_kq + koff128(kk), i128, kk > 0);
            umma_commit(&sc.bar_mma);
        }
        pend_mma = true;
        {
            // <dS', S> (the decay of the entering state into S'), from the hi + lo copy of dS'
            float p = 0.f;
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4) {
                const uint32_t off = sreg + sw128_off(r, sch + c4);
                const uint4 hv = *reinterpret_cast<const uint4*>(DST + off);
                const uint4 lv = *reinterpret_cast<const uint4*>(DSTLO + off);
                const uint32_t hw[4] = {hv.x, hv.y, hv.z, hv.w}, lw[4] = {lv.x, lv.y, lv.z, lv.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    p = fmaf(s32[8 * c4 + 2 * e], bf16_lo(hw[e]) + bf16_lo(lw[e]), p);
                    p = fmaf(s32[8 * c4 + 2 * e + 1], bf16_hi(hw[e]) + bf16_hi(lw[e]), p);
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
            if (lane == 0) sc.red[tid >> 5] = p;
        }
        wait_mma(ok);
        if (cg == 0) {
            // inverse norms from G's diagonal (rows past the chunk's tokens: 0)
            float d32[32];
            tmem_ld32(trow + T_G + static_cast<uint32_t>(r & ~31), d32);  // (warp-uniform columns)
            tmem_wait_ld();
            float nrm = 0.f;
#pragma unroll
            for (int e = 0; e < 32; ++e) nrm = (e == lane) ? d32[e] : nrm;
            const int row = r & 63;
            const float inv = row < n ? (a.l2norm ? 1.0f / sqrtf(nrm + 1e-6f) : 1.f) : 0.f;
            if (r < 64) sc.rk[row] = inv;
            else sc.rq[row] = inv;
        }
        __syncthreads();
        if (tid < 64) {
            const float bi = sc.bw[tid] + (tid >= 32 ? sc.bw[31] : 0.f);
            sc.b[tid] = bi;
            sc.gr[tid] = exp2f(bi) * sc.rk[tid];
        }
        __syncthreads();
        if (r >= 64) {
            // P = tril(scale rq_i rk_j (q_i . k_j) 2^{b_i - b_j}) in fp32 from G, hi + lo (MN-major B);
            // this thread: row i, columns 16 cg ..
            const int i = r - 64;
            float gq[16];
            tmem_ld16(trow + T_G + 16 * cg, gq);
            tmem_wait_ld();
            const float ci = a.scale * sc.rq[i], bi = sc.b[i];
            float pv[16], bj[16], rkj[16];
            ld8(bj, &sc.b[16 * cg]);
            ld8(bj + 8, &sc.b[16 * cg + 8]);
            ld8(rkj, &sc.rk[16 * cg]);
            ld8(rkj + 8, &sc.rk[16 * cg + 8]);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int j = 16 * cg + e;
                pv[e] = (i < n && j <= i) ? ci * rkj[e] * gq[e] * exp2f(bi - bj[e]) : 0.f;
            }
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                const uint32_t off = sw128_off(i, 2 * cg + c2);
                store8_split(PB + off, PLO + off, &pv[8 * c2]);
            }
        }

        // ---- P2: X^T = beta V^T - sx (.) (K S)^T -> hi, lo (this thread: value column r, tokens
        // 16 cg ..); then D^T = X^T T^T (T hi + lo) and (P^T dO)^T = dO^T P (P hi + lo)
        {
            float ks[16];
            tmem_ld16(trow + T_X1 + 16 * cg, ks);
            tmem_wait_ld();
            float x[16], bt[16], sxv[16];
            ld8(bt, &sc.bet[16 * cg]);
            ld8(bt + 8, &sc.bet[16 * cg + 8]);
            ld8(sxv, &sc.sx[16 * cg]);
            ld8(sxv + 8, &sc.sx[16 * cg + 8]);
#pragma unroll
            for (int e = 0; e < 16; ++e) x[e] = bt[e] * vv[e] - sxv[e] * ks[e];
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                const uint32_t off = sw128_off(r, 2 * cg + c2);
                store8_split(STLO + off, STLO + 16384 + off, &x[8 * c2]);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t i64 = idesc_bf16_f32(128, 64, false, false);
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_bf16(tmem + T_DT, d_xt + ((part * 16384) >> 4) + koff64(kk), d_tb + koff64(kk), i64,
                              (part | kk) != 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem + T_DT, d_xt + koff64(kk), d_tlo + koff64(kk), i64, 1u);
            const uint32_t imn = idesc_bf16_f32(128, 64, true, true);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem + T_ET, d_do_mn + moff(kk), d_p_mn + moff(kk), imn, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem + T_ET, d_do_mn + moff(kk), d_plo_mn + moff(kk), imn, 1u);
            umma_commit(&sc.bar_mma);
        }
        pend_mma = true;
        wait_mma(ok);

        // ---- P3: dD^T = (P^T dO)^T + sd (.) (K dS')^T -> hi, lo; D^T -> hi, lo; w; then dX^T = dD^T T
        {
            float d[16], e16[16], kd[16], sdv[16];
            tmem_ld16(trow + T_DT + 16 * cg, d);
            tmem_ld16(trow + T_ET + 16 * cg, e16);
            tmem_ld16(trow + T_X2 + 16 * cg, kd);
            ld8(sdv, &sc.sd[16 * cg]);
            ld8(sdv + 8, &sc.sd[16 * cg + 8]);
            tmem_wait_ld();
            float w[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const float k_ = sdv[e] * kd[e];
                w[e] = k_ * d[e];
                e16[e] += k_;
            }
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                const uint32_t off = sw128_off(r, 2 * cg + c2);
                store8_split(DSTLO + off, DSTLO + 16384 + off, &e16[8 * c2]);
                store8_split(STLO + off, STLO + 16384 + off, &d[8 * c2]);
            }
            const float ws = scatter_sum16(w, lane);
            if (lane < 16) sc.pw[q4][16 * cg + lane] = ws;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(!ok)) { failed = true; break; }
        if (tid == 0) {
            tc_fence_after();
            const uint32_t idy = idesc_bf16_f32(128, 64, false, true);
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    umma_bf16(tmem + T_DY, d_dd + ((part * 16384) >> 4) + koff64(kk), d_t_mn + moff(kk), idy,
                              (part | kk) != 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem + T_DY, d_dd + koff64(kk), d_tlo_mn + moff(kk), idy, 1u);
            umma_commit(&sc.bar_mma);
        }
        pend_mma = true;
        wait_mma(ok);

        // ---- P4: dV, the sums over the value columns, and the operands of the dA / dP and dk~ / dq~
        // products: [dX; dO] (MN-major, dX hi + lo), W = [-sx (.) dX | sq (.) dO]^T
        float dx[16], dov[16];
        {
            float ks[16], qs[16];
            tmem_ld16(trow + T_DY + 16 * cg, dx);
            tmem_ld16(trow + T_X1 + 16 * cg, ks);
            tmem_ld16(trow + T_X1 + 64 + 16 * cg, qs);
#pragma unroll
            for (int e = 0; e < 16; ++e) dov[e] = tile_col(DO, 8192, r, 16 * cg + e);
            float gr[16];
            ld8(gr, &sc.gr[16 * cg]);
            ld8(gr + 8, &sc.gr[16 * cg + 8]);
            tmem_wait_ld();
            float t16[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) t16[e] = dx[e] * (vv[e] - gr[e] * ks[e]);
            float s_ = scatter_sum16(t16, lane);
            if (lane < 16) sc.psb[q4][16 * cg + lane] = s_;
#pragma unroll
            for (int e = 0; e < 16; ++e) t16[e] = dx[e] * ks[e];
            s_ = scatter_sum16(t16, lane);
            if (lane < 16) sc.psg[q4][16 * cg + lane] = s_;
#pragma unroll
            for (int e = 0; e < 16; ++e) t16[e] = dov[e] * qs[e];
            s_ = scatter_sum16(t16, lane);
            if (lane < 16) sc.pso[q4][16 * cg + lane] = s_;
        }
        __syncthreads();  // the dO tile is read: its region takes the new operands
        {
            float sxv[16], sqv[16];
            ld8(sxv, &sc.sx[16 * cg]);
            ld8(sxv + 8, &sc.sx[16 * cg + 8]);
            ld8(sqv, &sc.sq[16 * cg]);
            ld8(sqv + 8, &sc.sq[16 * cg + 8]);
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
                const uint32_t off = sw128_off(r, 2 * cg + c2);
                store8_split(DSTLO + 16384 + off, DSTLO + off, &dx[8 * c2]);   // dX hi, lo
                store8_split(TLO + off, nullptr, &dov[8 * c2]);                  // dO (exact)
                float w0[8], w1[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    w0[e] = -sxv[8 * c2 + e] * dx[8 * c2 + e];
                    w1[e] = sqv[8 * c2 + e] * dov[8 * c2 + e];
                }
                store8_split(TB + off, nullptr, w0);
                store8_split(DO + off, nullptr, w1);
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(!ok)) { failed = true; break; }
        if (tid == 0) {
            tc_fence_after();
            const uint32_t imn = idesc_bf16_f32(128, 64, true, true);
            const uint64_t dlo = 16384 >> 4;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) umma_bf16(tmem + T_DAP, d_ax_mn + moff(kk), d_dt_mn + moff(kk), imn, kk > 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) umma_bf16(tmem + T_DAP, d_ax_mn + moff(kk), d_dt_mn + dlo + moff(kk), imn, 1u);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) umma_bf16(tmem + T_DAP2, d_axlo_mn + moff(kk), d_dt_mn + moff(kk), imn, kk > 0);
            umma_commit(&sc.bar_mma);  // dA / dP: the token-row phase starts while the rest runs
            // [dk~ ; dq~] = W^T S^T: token rows (A = W, MN-major), key columns (B = S^T, MN-major)
            const uint32_t ikq = idesc_bf16_f32(128, 128, true, true);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) umma_bf16(tmem + T_DKQ, d_w_mn + moff(kk), d_s_mn + moff(kk), ikq, kk > 0);
            umma_commit(&sc.bar_mma2);
        }
        pend_mma = pend_mma2 = true;
        wait_mma(ok);

        // ---- P5 (token rows): dA, dP with A, P recomputed from G; dbeta and db row / column
        // terms; N = diag(rk) M diag(rk) and Hs = diag(rq) H diag(rk) as bf16 tiles for the last products
        {
            const int i = r & 63;
            const bool isP = r >= 64;  // rows 64-127: dO D^T (else dX D^T)
            const bool rowv = i < n;
            const float bi = sc.b[i];
            const float ri = isP ? sc.rq[i] : sc.rk[i];
            const float beti = sc.bet[i];
            float rowsum = 0.f, sbsum = 0.f;
#pragma unroll 1
            for (int g = 0; g < 2; ++g) {
                const int j0 = 16 * cg + 8 * g;
                float dv8[8], gg[8];
                tmem_ld8(trow + T_DAP + j0, dv8);
                tmem_ld8(trow + T_G + j0, gg);
                if (!isP) {
                    float d2[8];
                    tmem_ld8(trow + T_DAP2 + j0, d2);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 8; ++e) dv8[e] += d2[e];
                } else {
                    tmem_wait_ld();
                }
                float colv[8], bj[8], rkj[8], tv[8];
                ld8(bj, &sc.b[j0]);
                ld8(rkj, &sc.rk[j0]);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int j = j0 + e;
                    float mval = 0.f, cv = 0.f;
                    if (rowv && (isP ? j <= i : j < i)) {
                        const float dec = exp2f(bi - bj[e]);
                        const float gk = ri * rkj[e] * gg[e] * dec;  // normalised, decayed (k_i . k_j) or (q_i . k_j)
                        if (isP) {
                            const float dP = dv8[e];
                            cv = dP * a.scale * gk;
                            mval = dP * a.scale * dec;
                        } else {
                            const float dA = -dv8[e];
                            sbsum = fmaf(dA, gk, sbsum);
                            cv = dA * beti * gk;
                            mval = dA * beti * dec;
                        }
                        rowsum += cv;
                    }
                    colv[e] = cv;
                    tv[e] = ri * mval * rkj[e];  // N_ij = rk_i M_ij rk_j, Hs_ij = rq_i H_ij rk_j
                }
                store8_split(NH + sw128_off(r, 2 * cg + g), nullptr, tv);
                const float cs = scatter_sum8(colv, lane);
                if (lane < 8) (isP ? sc.colP : sc.colA)[q4 & 1][j0 + lane] = cs;
            }
            if (isP) {
                sc.rowP[cg][i] = rowsum;
            } else {
                sc.rowA[cg][i] = rowsum;
                sc.sbA[cg][i] = sbsum;
            }
            // the zero tile the transposed reads of N and Hs take as their rows 64-127
            *reinterpret_cast<uint4*>(NH + 16384 + 16 * tid) = make_uint4(0u, 0u, 0u, 0u);
        }
        {
            // dk~ += W^T S^T has completed (the last products accumulate onto it)
            const bool ok2 = wait_phase(&sc.bar_mma2, ph_mma2, budget);
            if (ok2) {
                ph_mma2 ^= 1u;
                pend_mma2 = false;
            }
            ok = ok && ok2;
            // ... so S^T hi is read for the last time: the next item's S starts streaming into it
            const int64_t nx0 = item + static_cast<int64_t>(gridDim.x);
            if (ok2 && nx0 < total_items) {
                if (tid == kIo) load_state_half(nx0);
                pend_pre0 = true;
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == kMmaLast) {
            tc_fence_after();
            // acc2 = D dS'^T on the token rows (A = [D^T hi | D^T lo]: rows 64-127 unused; D hi only,
            // this term reaching only dk)
            const uint32_t imn = idesc_bf16_f32(128, 128, true, true);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) umma_bf16(tmem + T_ACC2, d_dt_mn + moff(kk), d_ds_mn + moff(kk), imn, kk > 0);
            // [dk~ ; dq~] += [N ; Hs] K  +  [N^T ; 0] K  +  [Hs^T ; 0] Q: the symmetric scalings make
            // the transposes plain MN-major reads of the same tiles (B: key or query rows, MN-major)
            const uint32_t ikm = idesc_bf16_f32(128, 128, false, true);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem + T_DKQ, d_nh + koff64(kk), d_kq_mn + moff(kk), ikm, 1u);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) umma_bf16(tmem + T_DKQ, d_nt_mn + moff(kk), d_kq_mn + moff(kk), imn, 1u);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                umma_bf16(tmem + T_DKQ, d_ht_mn + moff(kk), d_kq_mn + (8192 >> 4) + moff(kk), imn, 1u);
            umma_commit(&sc.bar_mma);
        }
        pend_mma = true;

        // ---- P7 (tokens, while the last product runs): dbeta, db, dg with the input transforms
        if (tid < 64) {
            const int j = tid;
            float dbeta = 0.f, db = 0.f;
            if (j < n) {
                dbeta = (sc.psb[0][j] + sc.psb[1][j] + sc.psb[2][j] + sc.psb[3][j]) +
                        ((sc.sbA[0][j] + sc.sbA[1][j]) + (sc.sbA[2][j] + sc.sbA[3][j]));
                const float sg = sc.psg[0][j] + sc.psg[1][j] + sc.psg[2][j] + sc.psg[3][j];
                const float so = sc.pso[0][j] + sc.pso[1][j] + sc.pso[2][j] + sc.pso[3][j];
                const float wj = sc.pw[0][j] + sc.pw[1][j] + sc.pw[2][j] + sc.pw[3][j];
                const float ra = (sc.rowA[0][j] + sc.rowA[1][j]) + (sc.rowA[2][j] + sc.rowA[3][j]);
                const float rp = (sc.rowP[0][j] + sc.rowP[1][j]) + (sc.rowP[2][j] + sc.rowP[3][j]);
                db = -sc.sx[j] * sg + sc.sq[j] * so + ra - (sc.colA[0][j] + sc.colA[1][j]) + rp -
                     (sc.colP[0][j] + sc.colP[1][j]) - wj;
            }
            // the chunk's total decay (of the entering state into S', and of the sd factors) at its
            // last token: w summed over the chunk by a warp reduction
            float wpart = 0.f;
            if (j < n) wpart = sc.pw[0][j] + sc.pw[1][j] + sc.pw[2][j] + sc.pw[3][j];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) wpart += __shfl_xor_sync(0xffffffffu, wpart, off);
            if (lane == 0) sc.gp[2 + (tid >> 5)] = wpart;
            asm volatile("bar.sync 1, 64;" ::: "memory");
            if (j == n - 1) {
                float ds = 0.f;
#pragma unroll
                for (int x = 0; x < 16; ++x) ds += sc.red[x];
                db += exp2f(sc.b[n - 1]) * ds + (sc.gp[2] + sc.gp[3]);
            }
            // dg_j = sum_{i >= j} db_i: suffix scans of the two warps, then the second warp's total
            float sacc = db;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float y = __shfl_down_sync(0xffffffffu, sacc, off);
                if (lane + off < 32) sacc += y;
            }
            sc.db[j] = sacc;
            asm volatile("bar.sync 1, 64;" ::: "memory");
            if (j < 32) sacc += sc.db[32];
            float pl = 0.f, pd = 0.f;
            if (j < n) {
                const int64_t t = t0 + j;
                float dgr = sacc, dbr = dbeta;
                if (a.gate_mode == LA_GATE_SOFTPLUS) {
                    const float z = a.g[t * a.g_st + h * a.g_sh] + gdt;
                    dgr = sacc * gAh / (1.f + expf(-z));
                    pl = sacc * sc.gt[j];
                    pd = dgr;
                } else if (a.gate_mode == LA_GATE_SIGMOID_BOUND) {
                    const float sx = 1.f / (1.f + expf(-a.g[t * a.g_st + h * a.g_sh]));
                    dgr = sacc * a.gate_lb * sx * (1.f - sx);
                }
                if (a.beta_sigmoid) dbr *= sc.bet[j] * (1.f - sc.bet[j]);
                bw.dg[t * bw.dg_st + h * bw.dg_sh] = dgr;
                bw.dbeta[t * bw.db_st + h * bw.db_sh] = dbr;
            }
            if (bw.gpart) {
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    pl += __shfl_xor_sync(0xffffffffu, pl, off);
                    pd += __shfl_xor_sync(0xffffffffu, pd, off);
                }
                asm volatile("bar.sync 1, 64;" ::: "memory");  // gp[] is free again
                if (lane == 0) {
                    sc.gp[2 * (tid >> 5)] = pl;
                    sc.gp[2 * (tid >> 5) + 1] = pd;
                }
                asm volatile("bar.sync 1, 64;" ::: "memory");
                if (tid == 0) {
                    // slot (head, chunk): the per-head sums then run over the chunks in order
                    const int64_t slot = static_cast<int64_t>(h) * bw.pieces + chunk;
                    bw.gpart[2 * slot] = sc.gp[0] + sc.gp[2];
                    bw.gpart[2 * slot + 1] = sc.gp[1] + sc.gp[3];
                }
            }
        }
        wait_mma(ok);
        fence_proxy_async_smem();  // (the prefetch below overwrites regions read and written by the threads)
        if (__syncthreads_or(!ok)) { failed = true; break; }
        {
            // the next item's S and dS' stream in while this one finishes: their regions are free
            const int64_t nx = item + static_cast<int64_t>(gridDim.x);
            prefetched = nx < total_items;
            if (tid == kIo && prefetched) load_states_rest(nx);
            pend_pre = prefetched;
            if (prefetched) item_meta(nx);
        }

        // ---- P6 (token rows): dk = dk~ - rk^2 (k . dk~) k, dq alike (thread: row r, 32 key columns
        // 32 cg ..; rows 0-63 dk, 64-127 dq), dk~ adding sd (.) acc2; then dv = beta (.) dX
        const bool full = n == kChunk && bw.out_tma != 0;
        {
            const int i = r & 63;
            const bool isq = r >= 64;
            float x[32];
            tmem_ld32(trow + T_DKQ + 32 * cg, x);
            if (!isq) {
                float y[32];
                tmem_ld32(trow + T_ACC2 + 32 * cg, y);
                tmem_wait_ld();
                const float sdi = sc.sd[i];
#pragma unroll
                for (int e = 0; e < 32; ++e) x[e] = fmaf(sdi, y[e], x[e]);
            } else {
                tmem_wait_ld();
            }
            if (a.l2norm) {
                // the raw row's columns (the K/Q tile: region cg / 2, row r, chunks 4 (cg % 2) ..)
                float kv[32];
                const uint8_t* row = KQ + (cg >> 1) * 16384;
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    const uint4 wv = *reinterpret_cast<const uint4*>(row + sw128_off(r, 4 * (cg & 1) + c4));
                    const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        kv[8 * c4 + 2 * e] = bf16_lo(ww[e]);
                        kv[8 * c4 + 2 * e + 1] = bf16_hi(ww[e]);
                    }
                }
                float pd = 0.f;
#pragma unroll
                for (int e = 0; e < 32; ++e) pd = fmaf(kv[e], x[e], pd);
                sc.pdot[cg][r] = pd;
                __syncthreads();
                const float rv = isq ? sc.rq[i] : sc.rk[i];
                const float cf = rv * rv * (((sc.pdot[0][r] + sc.pdot[1][r]) + sc.pdot[2][r]) + sc.pdot[3][r]);
#pragma unroll
                for (int e = 0; e < 32; ++e) x[e] = fmaf(-cf, kv[e], x[e]);
            }
            if (a.group == 1) {
                if (full) {
                    // staged for the TMA store: [column region][64 rows][128 B], swizzled
                    uint8_t* stg = (isq ? TLO : TB) + (cg >> 1) * 8192;
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) store8_split(stg + sw128_off(i, 4 * (cg & 1) + c4), nullptr, &x[8 * c4]);
                } else if (i < n) {
                    uint16_t* o = (isq ? bw.dq + (t0 + i) * bw.dq_st + hk * bw.dq_sh
                                       : bw.dk + (t0 + i) * bw.dk_st + hk * bw.dk_sh) + 32 * cg;
                    if (bw.vec_out) {
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4) store8_split(reinterpret_cast<uint8_t*>(o + 8 * c4), nullptr, &x[8 * c4]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = f_to_bf16_bits(x[e]);
                    }
                }
            } else if (i < n) {
                float* o = (isq ? bw.dqh : bw.dkh) + ((t0 + i) * HO + h) * KD + 32 * cg;
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4)
                    *reinterpret_cast<float4*>(o + 4 * c4) = make_float4(x[4 * c4], x[4 * c4 + 1], x[4 * c4 + 2], x[4 * c4 + 3]);
            }
        }
        {
            // dv = beta (.) dX (still in TMEM): value column r, tokens 16 cg ..
            uint8_t* stg = DO + (r >> 6) * 8192 + (r & 7) * 2;
            const uint32_t sck = static_cast<uint32_t>((r & 63) >> 3);
            uint16_t* dvp = bw.dv + h * bw.dv_sh + r;
#pragma unroll 1
            for (int g = 0; g < 2; ++g) {
                float d8[8], bt[8];
                tmem_ld8(trow + T_DY + 16 * cg + 8 * g, d8);
                ld8(bt, &sc.bet[16 * cg + 8 * g]);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int i = 16 * cg + 8 * g + e;
                    const uint16_t val = f_to_bf16_bits(bt[e] * d8[e]);
                    if (full) *reinterpret_cast<uint16_t*>(stg + sw128_off(static_cast<uint32_t>(i), sck)) = val;
                    else if (i < n) dvp[(t0 + i) * bw.dv_st] = val;
                }
            }
        }
        if (full) {
            fence_proxy_async_smem();
            __syncthreads();
            if (tid == kIo) {
#pragma unroll
                for (int rg = 0; rg < 2; ++rg) {
                    tma_store_3d(&dvmap, DO + rg * 8192, rg * 64, h, static_cast<int>(t0));
                    if (a.group == 1) {
                        tma_store_3d(&dkmap, TB + rg * 8192, rg * 64, hk, static_cast<int>(t0));
                        tma_store_3d(&dqmap, TLO + rg * 8192, rg * 64, hk, static_cast<int>(t0));
                    }
                }
                bulk_commit_group();
            }
        }
        tc_fence_before();
        __syncthreads();  // every read of this item's tiles and TMEM is done
    }

    if (failed) {
        // let in-flight copies and products finish (bounded) before TMEM and shared memory go away
        if (pend_in) wait_phase(&sc.bar_in, ph_in, budget);
        if (pend_pre) wait_phase(&sc.bar_pre, ph_pre, budget);
        if (pend_pre0) wait_phase(&sc.bar_pre0, ph_pre0, budget);
        if (pend_mma) wait_phase(&sc.bar_mma, ph_mma, budget);
        if (pend_mma2) wait_phase(&sc.bar_mma2, ph_mma2, budget);
        if (tid == 0) {
            atomicCAS(&a.hdr->status, LA_OK, LA_ERR_TIMEOUT);
            if (a.user_status) atomicCAS(a.user_status, LA_OK, LA_ERR_TIMEOUT);
        }
    }
    if (tid == kIo) bulk_wait_all();  // the last output tiles are out before the CTA ends
    tc_fence_before();
    __syncthreads();
    if (tid < 32) tmem_dealloc(tmem, T_COLS);
}

}  // namespace

cudaError_t launch_dchunk(const ChunkArgs& a, const BwdArgs& b, const CUtensorMap& qm, const CUtensorMap& km,
                          const CUtensorMap& dom, const CUtensorMap& wm, const CUtensorMap& dkm, const CUtensorMap& dqm,
                          const CUtensorMap& dvm, cudaStream_t s) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gdn_dchunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(D_SMEM));
    if (e != cudaSuccess) return e;
    // one CTA per SM (the whole tensor memory and ~226 KB of shared memory), persistent over the
    // (chunk, head) items; a.items bounds them (the prologue's chunk count decides)
    const int64_t grid = a.items < sms ? a.items : sms;
    if (grid <= 0) return cudaSuccess;
    gdn_dchunk_kernel<<<static_cast<int>(grid), kDT, D_SMEM, s>>>(qm, km, dom, wm, dkm, dqm, dvm, a, b);
    return cudaGetLastError();
}

}  // namespace la
