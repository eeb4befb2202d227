// gdn_kernel.h -- internal interface between the C ABI (la_api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace la {

constexpr int kChunk = 64;          // tokens per chunk; the chunk grid restarts at each sequence
constexpr int kThreads = 256;       // threads of the fused chunk kernel
constexpr int kPrologueThreads = 1024;

// kModeGdp: the forward of Gated DeltaProduct (n delta updates per token) on the update timeline,
// with q, g and o on the token timeline.  kModeFwdSplit / kModeSummarySplit / kModeGdpSplit:
// the forward's, the summary's or GDP's state pass, reading each chunk's T (and P) and per-token
// factors from the records the WY pass (gdn_wy_kernel) wrote.
enum Mode : int {
    kModeFwd = 0, kModeSummary = 1, kModeGdp = 2, kModeFwdSplit = 3, kModeSummarySplit = 4, kModeGdpSplit = 5
};
enum TileKind : int { kTileValue = 0, kTileTransition = 1 };

// Workspace layout (bytes from the 256-aligned workspace base).
//   [0, 256)                 header: status, ticket
//   [256, 256 + 4N)          order[N]: sequences sorted longest-first (ties by index)
//   next 256-aligned, 8N     ckpt_off[N]: first checkpoint row of each sequence
//   next 256-aligned, 8P     sort keys (P = next power of two >= N), used only when N is
//                            too large for the prologue's shared-memory sort
struct WorkspaceLayout {
    size_t order, ckpt_off, keys, total;
};
__host__ __device__ inline size_t ws_align(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
__host__ __device__ inline uint32_t next_pow2(uint32_t n) {
    uint32_t p = 1;
    while (p < n) p <<= 1;
    return p;
}
constexpr uint32_t kSmemSortMax = 8192;  // keys sorted in shared memory up to this many
__host__ __device__ inline WorkspaceLayout ws_layout(int32_t N) {
    WorkspaceLayout L;
    const size_t n = N > 0 ? static_cast<size_t>(N) : 1;
    L.order = 256;
    L.ckpt_off = ws_align(L.order + 4 * n);
    L.keys = ws_align(L.ckpt_off + 8 * n);
    const size_t p = n > kSmemSortMax ? next_pow2(static_cast<uint32_t>(n)) : 0;
    L.total = ws_align(L.keys + 8 * p);
    return L;
}

// The two-pass forward's extra workspace, after ws_layout(N): chunk_off[N + 1] (each
// sequence's first chunk in the batch-wide chunk numbering, and the total), chunk_seq[chunks]
// (the sequence of each chunk), then one WY record
// per (chunk, head) item, item = chunk * HV + h: T (bf16 [64][64], row-major), P (bf16
// [64][64]) and the factors beta, sx, sq, sd (fp32 [4][64]).  A batch has at most T / 64 + N
// chunks.
constexpr size_t kWyTileBytes = 64 * 64 * 2;
constexpr size_t kWyFactorBytes = 4 * 64 * 4;
constexpr size_t kWyRecordBytes = 2 * kWyTileBytes + kWyFactorBytes;  // 17408: 136 rows of 128 B
struct SplitLayout {
    size_t chunk_off, chunk_seq, wy, total;
    int64_t chunks, items;
};
__host__ __device__ inline SplitLayout split_layout(int64_t T, int32_t N, int32_t HV) {
    SplitLayout L;
    const size_t n = N > 0 ? static_cast<size_t>(N) : 1;
    L.chunks = T / kChunk + (N > 0 ? N : 0);
    L.items = L.chunks * static_cast<int64_t>(HV > 0 ? HV : 0);
    L.chunk_off = ws_layout(N).total;
    L.chunk_seq = ws_align(L.chunk_off + 8 * (n + 1));
    L.wy = ws_align(L.chunk_seq + 4 * static_cast<size_t>(L.chunks > 0 ? L.chunks : 1));
    L.total = ws_align(L.wy + static_cast<size_t>(L.items) * kWyRecordBytes);
    return L;
}

struct WsHeader {
    int32_t status;     // LA_OK or a device-side error code
    int32_t ckpt_rows;  // sum_i ceil(L_i / n) when the prologue computed checkpoint offsets
    uint64_t ticket;    // next unit to hand out (8-byte aligned for the 64-bit atomic)
    int32_t ranges_ok;  // the sequences' chunk counts are within 1/8 of each other (forward ranges pay)
    int32_t reserved;
    int64_t total_chunks;  // sum_i ceil(L_i / 64) when the prologue computed chunk offsets
    uint64_t wy_ticket;    // next WY item to hand out
};
static_assert(sizeof(WsHeader) <= 256, "the header lives in the workspace's first 256 bytes");

struct PrologueArgs {
    const void* cu;
    int32_t cu64;
    int64_t T;
    int32_t N;
    int64_t ckpt_n;       // 0: no checkpoint offsets
    WsHeader* hdr;
    int32_t* order;
    int64_t* ckpt_off;
    uint64_t* keys;       // global sort scratch (N > kSmemSortMax)
    int32_t* user_status; // nullable
    int64_t* chunk_off;   // nullable: [N + 1] first chunk of each sequence, then the total
    int32_t chunk_rows;   // rows per token on the chunked timeline (GDP: its updates per token; else 1)
    int32_t* chunk_seq;   // with chunk_off: [total] the sequence of each chunk
};

struct ChunkArgs {
    // per-token scalars [T, HO]
    const float* g;
    int64_t g_st, g_sh;
    const float* beta;
    int64_t b_st, b_sh;
    const void* cu;
    int32_t cu64;
    int64_t T;
    int32_t N, HK, HV, K, V, group;  // group = HV / HK
    float scale;
    int32_t l2norm;
    const void* s0;                  // [N, HO, K, V] or null
    int32_t s0_bf16;
    uint16_t* o;                     // [T, HO, V] bf16 bits (fwd)
    int64_t o_st, o_sh;
    int32_t o_tma;                   // o is 16-byte aligned with strides in 16-byte units: full chunks go out by TMA
    float* final_state;              // fwd: final state; summary: end state
    void* ckpt;                      // [R, HO, K, V]
    int32_t ckpt_bf16;
    int64_t ckpt_n;
    float* transition;               // summary: [N, HO, K, K]
    int32_t tiles_per_head;          // fwd 1; summary 2 (value tile, transition tile)
    int64_t num_units;               // N * HO * tiles_per_head
    // Summary with more units than one wave, or a forward (fp32 final state) with one to four
    // waves of units: each unit's chunks run as `pieces` consecutive ranges in successive
    // launches (items r * num_units + u, range r of unit u); this launch's CTA b runs item
    // item_base + b.  A range starts from the state the previous range left in the outputs (end
    // or final state, transition).  pieces 1: one persistent launch over the units.
    int32_t pieces;
    int32_t pieces_request;          // forward: 0 automatic, 1 whole walks, >= 2 that many ranges (test hook)
    // A forward launched in automatic ranges still walks whole sequences when the prologue found
    // their lengths spread (WsHeader::ranges_ok = 0): the first launch then runs the persistent
    // walk over whole units and the later launches return at once.
    int64_t item_base;
    int64_t items;                   // items of this launch
    WsHeader* hdr;
    const int32_t* order;
    const int64_t* ckpt_off;
    int32_t* user_status;
    uint64_t wait_budget_ns;
    int32_t test_skip_tile_load;     // failure-path test: never load K/Q tiles, so the first wait runs out
    // optional input transforms (la_gate_mode, beta logits)
    int32_t gate_mode;
    const float* a_log;              // [HO]
    const float* dt_bias;            // [HO]
    float gate_lb;
    int32_t beta_sigmoid;
    int32_t beta_bf16;
    int32_t gdp_n;                   // kModeGdp: updates per token (divides 64); k, v, beta have n rows per token
    // state pool: sequence i reads and writes back slot state_idx[i] of s0 (then final_state
    // aliases s0 and final_bf16 follows the pool's dtype)
    const int32_t* state_idx;
    int64_t pool_size;
    int32_t final_bf16;
    // the two-pass forward (kModeFwdSplit and the WY pass): chunk offsets and the WY records
    const int64_t* chunk_off;
    const int32_t* chunk_seq;
    uint8_t* wy;
    // the state-gradient pass of gdn_bwd: the gradient of the state leaving every chunk, per
    // (chunk, head) item, as the bf16 hi and lo parts of dS^T [2][128 rows][128 B] (64 KB), or null
    uint8_t* ds_chunks;
    // the WY pass for gdn_bwd also writes T's bf16 residual per item (8 KB, swizzled), or null
    uint8_t* wy_tlo;
    // the state-gradient pass of gdn_bwd when its units outnumber the SMs: each unit's chunks in
    // `pieces` ranges taken in dependency order by co-resident CTAs, a range starting from the
    // gradient its successor left here ([N * HO][K][V] fp32) once the unit's flag says so
    float* grad_carry;
    int32_t* grad_flags;             // [N * HO], zeroed by the launch
};

// One recurrence step per sequence against a state pool (gdn_decode).
struct DecodeArgs {
    const uint16_t* q; int64_t q_sn, q_sh;
    const uint16_t* k; int64_t k_sn, k_sh;
    const uint16_t* v; int64_t v_sn, v_sh;
    const float* g; int64_t g_sn, g_sh;
    const void* beta; int64_t b_sn, b_sh;
    int32_t N, HK, HV, K, V, group;
    float scale;
    int32_t l2norm;
    void* pool;                      // [pool_size, HV, K, V], updated in place
    int32_t pool_bf16;
    int64_t pool_size;
    const int32_t* idx;              // [N] or null (sequence i uses slot i)
    uint16_t* o; int64_t o_sn, o_sh;
    int32_t* status;                 // nullable
    int32_t gate_mode;
    const float* a_log;
    const float* dt_bias;
    float gate_lb;
    int32_t beta_sigmoid;
    int32_t beta_bf16;
};

// The backward (gdn_bwd): one CTA per (sequence, head), reverse over chunks.
struct BwdArgs {
    const uint16_t* q; int64_t q_st, q_sh;
    const uint16_t* k; int64_t k_st, k_sh;
    const uint16_t* v; int64_t v_st, v_sh;
    const float* g; int64_t g_st, g_sh;
    const float* beta; int64_t b_st, b_sh;
    const void* cu;
    int32_t cu64;
    int64_t T;
    int32_t N, HK, HV, K, V, group;
    float scale;
    int32_t l2norm;
    const uint16_t* dout; int64_t do_st, do_sh;
    const float* dfinal;             // [N, HO, K, V] or null
    const float* ckpt;               // states entering every chunk, [rows, HO, K, V] fp32
    const int64_t* ckpt_off;         // [N] first chunk row of each sequence
    const WsHeader* hdr;             // the prologue's status word: nothing runs unless LA_OK
    float* dS_work;                  // [N * HO, K, V]
    uint16_t* dq; int64_t dq_st, dq_sh;
    uint16_t* dk; int64_t dk_st, dk_sh;
    uint16_t* dv; int64_t dv_st, dv_sh;
    float* dg; int64_t dg_st, dg_sh;
    float* dbeta; int64_t db_st, db_sh;
    float* ds0;                      // [N, HO, K, V] or null
    float* dqh;                      // [T, HO, K] fp32 per value head (grouped heads)
    float* dkh;
    int32_t vec_out;                 // dq, dk rows 16-byte aligned: 16-byte stores
    int32_t vo_async;                // v, dO pairs 4-byte aligned: asynchronous 4-byte copies
    int32_t out_tma;                 // dq, dk, dv rows 16-byte aligned with strides in 16-byte units:
                                     // the tensor-core pass stores full chunks by TMA
    int32_t state_only;              // only the entering-state gradient (gdn_summary_bwd): no
                                     // checkpoints, v, dq, dk, dv, dg, dbeta
    // input transforms as in the forward; dg, dbeta then refer to the raw inputs
    int32_t gate_mode;               // la_gate_mode
    const float* a_log;              // [HO] (LA_GATE_SOFTPLUS)
    const float* dt_bias;            // [HO] (LA_GATE_SOFTPLUS)
    float gate_lb;                   // (LA_GATE_SIGMOID_BOUND)
    int32_t beta_sigmoid;            // beta holds logits
    int32_t beta_bf16;               // beta is bf16
    float* gpart;                    // [N * HO][pieces][2] per-piece sums for d_a_log, d_dt_bias, or null
    float* d_a_log;                  // [HO] or null
    float* d_dt_bias;                // [HO] or null
    // A unit's chunks are cut into `pieces` consecutive ranges run in reverse order by successive
    // launches; this launch's CTA b runs work item item_base + b (pieces 1: one item per unit).
    int32_t pieces;
    int32_t item_base;
};
constexpr int kBwdPieces = 4;

// Gated DeltaProduct: the update timeline for the chunk kernel, and the per-token outputs.
struct GdpArgs {
    int64_t T;                       // tokens
    int32_t N, HK, HO, K, V, n;      // n updates per token
    const uint16_t* q; int64_t q_st, q_sh;
    const float* g; int64_t g_st, g_sh;
    const void* cu;
    int32_t cu64;
    int32_t gate_mode;
    const float* a_log;
    const float* dt_bias;
    float gate_lb;
    uint16_t* qe;                    // [T * n, HK, K] contiguous
    float* ge;                       // [T * n, HO] contiguous
    int64_t* cue;                    // [N + 1]
    const uint16_t* oe;              // [T * n, HO, V] contiguous
    uint16_t* o; int64_t o_st, o_sh;
};

// Checkpoint rows for the backward (gdn_ckpt.cu).  widen: the first hdr->ckpt_rows rows (at most
// max_rows) of bf16 checkpoints to fp32.  segments: the pseudo-sequences that cut every sequence
// at multiples of n (cu_seg [max_seg + 1], int64; trailing entries empty) and their start states
// (s0_seg [max_seg][row_elems] fp32: the given rows, zero beyond them), from the cadence-n
// checkpoint offsets a prologue wrote (ckpt_off_n, hdr_n).
struct CkptArgs {
    const void* src;        // given checkpoint rows (fp32 or bf16)
    int32_t src_bf16;
    int64_t row_elems;      // HO * K * V
    const WsHeader* hdr;    // rows and status from the prologue
    int64_t max_rows;
    float* dst;             // widen: fp32 rows
    const void* cu;         // segments: the batch's cu_seqlens
    int32_t cu64;
    int32_t N;
    int64_t T;
    int64_t n;
    const int64_t* ckpt_off_n;
    int64_t* cu_seg;
    float* s0_seg;
    int64_t max_seg;
};
cudaError_t launch_ckpt_widen(const CkptArgs& a, cudaStream_t s);
cudaError_t launch_ckpt_segments(const CkptArgs& a, cudaStream_t s);

// Launchers (return cudaError_t of the launch).
cudaError_t launch_gdp_expand(const GdpArgs& a, cudaStream_t s);
cudaError_t launch_gdp_gather(const GdpArgs& a, cudaStream_t s);
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_bwd(const BwdArgs& a, cudaStream_t s);
// After the chunk-parallel gradient pass: the sums over grouped value heads (dqh, dkh -> dq, dk)
// and the gate-parameter sums (gpart, N x HV x pieces slots, added in slot order).
cudaError_t launch_bwd_finish(const BwdArgs& a, cudaStream_t s);
cudaError_t launch_prologue(const PrologueArgs& a, cudaStream_t s);
// Composition of span summaries (gdn_compose_spans): out [R + 1, HO, K, V].
struct ComposeArgs {
    int32_t R, HO, K, V;
    const float* transitions;  // [R, HO, K, K]
    const float* terms;        // [R, HO, K, V]
    const float* start;        // [HO, K, V] or null (zeros)
    float* out;
    int32_t backward;
};
cudaError_t launch_compose(const ComposeArgs& a, cudaStream_t s);

// The WY pass of the two-pass forward or summary: one record per (chunk, head) item (wymap: the
// records as [items][136 rows][64] bf16); summary: the records without P.
// The state-gradient pass of gdn_summary_bwd on the WY records (a.s0: the gradient leaving each
// span or null, a.final_state: the gradient entering it; domap: dO as [T][HV][V] bf16).
cudaError_t launch_grad(const ChunkArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                        const CUtensorMap& domap, const CUtensorMap& wymap, cudaStream_t s);
// The chunk-parallel gradient pass of gdn_bwd (K = V = 128): per (chunk, head) item, from the
// entering state (bw.ckpt, fp32 at the chunk cadence), the stored leaving-state gradient
// (a.ds_chunks), the WY record and T's residual (a.wy_tlo), the gradients dq, dk (or the per-value-head dqh, dkh), dv,
// dg, dbeta and the per-item gate-parameter sums (bw.gpart, slot head * bw.pieces + chunk).
cudaError_t launch_dchunk(const ChunkArgs& a, const BwdArgs& bw, const CUtensorMap& qmap, const CUtensorMap& kmap,
                          const CUtensorMap& domap, const CUtensorMap& wymap, const CUtensorMap& dkmap,
                          const CUtensorMap& dqmap, const CUtensorMap& dvmap, cudaStream_t s);
enum WyKind : int { kWyFwd = 0, kWySummary = 1, kWyGdp = 2 };
cudaError_t launch_wy_kernel(const ChunkArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                             const CUtensorMap& wymap, int kind, cudaStream_t s);
cudaError_t launch_chunk_kernel(const ChunkArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, const CUtensorMap& omap, const CUtensorMap& wymap, int mode,
                                cudaStream_t s);
int chunk_kernel_grid(int device, int64_t num_units);

}  // namespace la
