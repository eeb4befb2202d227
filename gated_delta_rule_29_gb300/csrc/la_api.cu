// la_api.cu -- the extern "C" boundary of liblinattn (declared in include/liblinattn.h).
//
// Host work only: argument validation (metadata, never values), TMA descriptor
// encoding from the caller's strides, workspace selection, and two launches on
// the caller's stream: the device prologue and the fused chunk kernel.  No host
// synchronisation happens on this path.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>

#include "../../include/liblinattn.h"
#include "gdn_kernel.h"

namespace {

using la::ChunkArgs;
using la::PrologueArgs;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

constexpr uint64_t kWaitBudgetNs = 1000000000ull;  // 1 s per bounded wait

// Events recorded around the next chunk-kernel launch of this host thread.
thread_local cudaEvent_t t_timing_start = nullptr;
thread_local cudaEvent_t t_timing_stop = nullptr;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// [T, H, D] bf16 view with 64 x 1 x 64 boxes (64 features of one head, 64 tokens), 128-byte swizzle.
la_status make_map(CUtensorMap* m, const void* base, int64_t T, int64_t H, int64_t D, int64_t st, int64_t sh,
                   uint32_t box_rows = 64) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return LA_ERR_CUDA;
    if (H == 1) sh = D;  // the stride of a size-1 axis is never used
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(sh) * 2, static_cast<cuuint64_t>(st) * 2};
    cuuint32_t box[3] = {64, 1, box_rows};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? LA_OK : LA_ERR_INVALID_ARG;
}

// A bf16 [T, H, D] operand read through TMA: 16-byte base, strides multiples of 8 elements.
la_status check_tma_operand(const void* p, int64_t st, int64_t sh, int64_t H) {
    if (!p) return LA_ERR_INVALID_ARG;
    if (!aligned(p, 16)) return LA_ERR_INVALID_ARG;
    if (st <= 0 || st % 8 != 0) return LA_ERR_INVALID_ARG;
    if (H > 1 && (sh <= 0 || sh % 8 != 0)) return LA_ERR_INVALID_ARG;
    return LA_OK;
}

struct DeviceWorkspace {
    void* ptr = nullptr;
    size_t bytes = 0;
};
std::mutex g_ws_mutex;
DeviceWorkspace g_ws[128];

// Internal per-device workspace, grown on demand without synchronising anything: a larger
// buffer replaces the current one and the old buffer is kept allocated until the process exits
// (kernels enqueued earlier, on any stream, may still be reading it, and freeing it safely would
// need a device-wide synchronisation).  Sizes at least double, so the kept buffers add up to
// less than the current one.  Growth allocates, which a stream capture does not allow: a call
// on a capturing stream that would need a larger buffer returns LA_ERR_WORKSPACE (nothing is
// launched; pass a workspace, or make one call of that size before capturing).
la_status internal_workspace(size_t need, cudaStream_t stream, void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return LA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    DeviceWorkspace& w = g_ws[dev];
    if (w.bytes < need) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return LA_ERR_CUDA;
        if (cs != cudaStreamCaptureStatusNone) return LA_ERR_WORKSPACE;
        size_t grow = 2 * w.bytes;
        if (grow < need) grow = need;
        if (grow < (size_t(1) << 20)) grow = size_t(1) << 20;
        void* p = nullptr;
        if (cudaMalloc(&p, grow) != cudaSuccess) {
            (void)cudaGetLastError();  // an allocation failure must not surface as a later launch error
            return LA_ERR_CUDA;
        }
        w.ptr = p;  // the previous buffer, if any, stays allocated (see above)
        w.bytes = grow;
    }
    *out = w.ptr;
    return LA_OK;
}

// Failure-path test hooks, set only through la_test_set_wait_hooks (never from the
// environment): skip the forward's K/Q tile loads, and replace the bounded waits' budget.
std::atomic<int32_t> g_test_skip_tile_load{0};
std::atomic<uint64_t> g_test_wait_budget_ns{0};
// Scheduling test hooks, set only through la_test_set_fwd_pieces / la_test_set_fwd_passes:
// 0 automatic chunk ranges; 0 automatic choice of the fused or the two-pass forward.
std::atomic<int32_t> g_test_fwd_pieces{0};
std::atomic<int32_t> g_test_fwd_passes{0};

la_status resolve_workspace(void* user, size_t user_bytes, int32_t N, cudaStream_t stream, void** out) {
    const size_t need = la::ws_layout(N).total;
    if (user) {
        if (user_bytes < need || !aligned(user, 256)) return LA_ERR_WORKSPACE;
        *out = user;
        return LA_OK;
    }
    return internal_workspace(need, stream, out);
}

struct Common {
    int64_t T;
    int32_t N, HK, HV, K, V;
    const void* cu;
    int32_t cu_bits;
    const float* g;
    const float* beta;
    int32_t beta_bytes;  // 4 (fp32) or 2 (bf16)
};

// The optional input transforms (cudnn-frontend PR #616: in-kernel softplus / bounded gate,
// beta sigmoid); validated here, applied by the chunk kernel as it loads g and beta.
la_status set_transforms(ChunkArgs& ka, int32_t gate_mode, const float* a_log, const float* dt_bias, float lb,
                         int32_t beta_sigmoid, int32_t beta_bf16) {
    if (gate_mode == LA_GATE_SOFTPLUS) {
        if (!a_log || !dt_bias || !aligned(a_log, 4) || !aligned(dt_bias, 4)) return LA_ERR_INVALID_ARG;
    } else if (gate_mode == LA_GATE_SIGMOID_BOUND) {
        if (!(lb < 0.f) || !std::isfinite(lb)) return LA_ERR_INVALID_ARG;
    } else if (gate_mode != LA_GATE_LOG) {
        return LA_ERR_INVALID_ARG;
    }
    ka.gate_mode = gate_mode;
    ka.a_log = gate_mode == LA_GATE_SOFTPLUS ? a_log : nullptr;
    ka.dt_bias = gate_mode == LA_GATE_SOFTPLUS ? dt_bias : nullptr;
    ka.gate_lb = lb;
    ka.beta_sigmoid = beta_sigmoid != 0;
    ka.beta_bf16 = beta_bf16 != 0;
    return LA_OK;
}

// The same transforms for the backward kernel's arguments.
la_status set_bwd_transforms(la::BwdArgs& b, int32_t gate_mode, const float* a_log, const float* dt_bias, float lb,
                             int32_t beta_sigmoid, int32_t beta_bf16) {
    ChunkArgs ka;
    std::memset(&ka, 0, sizeof(ka));
    const la_status st = set_transforms(ka, gate_mode, a_log, dt_bias, lb, beta_sigmoid, beta_bf16);
    if (st != LA_OK) return st;
    b.gate_mode = ka.gate_mode;
    b.a_log = ka.a_log;
    b.dt_bias = ka.dt_bias;
    b.gate_lb = ka.gate_lb;
    b.beta_sigmoid = ka.beta_sigmoid;
    b.beta_bf16 = ka.beta_bf16;
    return LA_OK;
}

la_status check_common(const Common& c) {
    if (c.T < 0 || c.N < 0 || c.HK <= 0 || c.HV <= 0) return LA_ERR_INVALID_ARG;
    if (c.cu_bits != 32 && c.cu_bits != 64) return LA_ERR_INVALID_ARG;
    if (!c.cu || !aligned(c.cu, c.cu_bits / 8)) return LA_ERR_INVALID_ARG;
    if ((c.K != 64 && c.K != 128) || (c.V != 64 && c.V != 128)) return LA_ERR_UNSUPPORTED;
    if (c.HV % c.HK != 0) return LA_ERR_UNSUPPORTED;
    if (c.T >= (int64_t(1) << 31) - 64) return LA_ERR_UNSUPPORTED;  // TMA coordinates are int32
    if (c.T > 0 && (!c.g || !c.beta || !aligned(c.g, 4) || !aligned(c.beta, c.beta_bytes))) return LA_ERR_INVALID_ARG;
    return LA_OK;
}

// gdp_n > 1 (mode kModeGdp): k, v (and beta) have gdp_n rows per token, q, g and o one; the q and
// o tiles then hold 64 / gdp_n token rows per 64-row chunk.
la_status run(const Common& c, ChunkArgs& ka, const void* q, int64_t q_st, int64_t q_sh, const void* k, int64_t k_st,
              int64_t k_sh, const void* v, int64_t v_st, int64_t v_sh, int64_t ckpt_n, void* workspace,
              size_t workspace_bytes, int32_t* user_status, int mode, cudaStream_t stream, int32_t gdp_n = 1) {
    void* ws = nullptr;
    // The forward and the summary run as two passes (the WY pass over every (chunk, head), then
    // the state pass) when the workspace has room for the WY records; otherwise as the fused
    // kernel.  Both give the same bits.
    const int32_t passes = g_test_fwd_passes.load(std::memory_order_relaxed);
    const la::SplitLayout SL = la::split_layout(c.T * gdp_n, c.N, c.HV);
    bool split = (mode == la::kModeFwd || mode == la::kModeSummary || mode == la::kModeGdp) && c.T > 0 &&
                 passes != 1 && SL.items < (int64_t(1) << 31);
    la_status st = LA_OK;
    if (split) {
        if (workspace) {
            split = workspace_bytes >= SL.total && aligned(workspace, 256);
            if (split) ws = workspace;
        } else {
            split = internal_workspace(SL.total, stream, &ws) == LA_OK;
        }
    }
    if (!split && (st = resolve_workspace(workspace, workspace_bytes, c.N, stream, &ws)) != LA_OK) return st;
    const la::WorkspaceLayout L = la::ws_layout(c.N);
    uint8_t* wsb = static_cast<uint8_t*>(ws);

    PrologueArgs pa;
    pa.cu = c.cu;
    pa.chunk_off = split ? reinterpret_cast<int64_t*>(wsb + SL.chunk_off) : nullptr;
    pa.chunk_seq = split ? reinterpret_cast<int32_t*>(wsb + SL.chunk_seq) : nullptr;
    pa.chunk_rows = gdp_n;
    pa.cu64 = c.cu_bits == 64;
    pa.T = c.T;
    pa.N = c.N;
    pa.ckpt_n = ckpt_n;
    pa.hdr = reinterpret_cast<la::WsHeader*>(wsb);
    pa.order = reinterpret_cast<int32_t*>(wsb + L.order);
    pa.ckpt_off = reinterpret_cast<int64_t*>(wsb + L.ckpt_off);
    pa.keys = reinterpret_cast<uint64_t*>(wsb + L.keys);
    pa.user_status = user_status;
    if (la::launch_prologue(pa, stream) != cudaSuccess) return LA_ERR_CUDA;

    const int32_t HO = c.HV;
    ka.g = c.g;
    ka.beta = c.beta;
    ka.cu = c.cu;
    ka.cu64 = c.cu_bits == 64;
    ka.T = c.T;
    ka.N = c.N;
    ka.HK = c.HK;
    ka.HV = c.HV;
    ka.K = c.K;
    ka.V = c.V;
    ka.group = c.HV / c.HK;
    ka.num_units = static_cast<int64_t>(c.N) * HO * ka.tiles_per_head;
    ka.hdr = pa.hdr;
    ka.order = pa.order;
    ka.ckpt_off = pa.ckpt_off;
    ka.user_status = user_status;
    ka.wait_budget_ns = kWaitBudgetNs;
    // failure-path test hooks (off unless a test set them with la_test_set_wait_hooks)
    ka.test_skip_tile_load = g_test_skip_tile_load.load(std::memory_order_relaxed) != 0;
    if (const uint64_t b = g_test_wait_budget_ns.load(std::memory_order_relaxed)) ka.wait_budget_ns = b;
    ka.pieces_request = g_test_fwd_pieces.load(std::memory_order_relaxed);
    ka.chunk_off = pa.chunk_off;
    ka.chunk_seq = pa.chunk_seq;
    ka.wy = split ? wsb + SL.wy : nullptr;
    if (ka.num_units == 0) return LA_OK;

    CUtensorMap qm, km, vm, om, wm;
    std::memset(&qm, 0, sizeof(qm));
    std::memset(&km, 0, sizeof(km));
    std::memset(&vm, 0, sizeof(vm));
    std::memset(&om, 0, sizeof(om));
    std::memset(&wm, 0, sizeof(wm));
    // the WY records as [items][136 rows][64] bf16: T at row 0, P at row 64 (the factors follow)
    if (split && (st = make_map(&wm, ka.wy, 136, SL.items, 64, 64, static_cast<int64_t>(la::kWyRecordBytes / 2))) !=
                     LA_OK)
        return st;
    const int64_t Tm = c.T > 0 ? c.T : 1;  // descriptors need a non-empty extent
    const uint32_t qrows = static_cast<uint32_t>((la::kChunk + gdp_n - 1) / gdp_n);
    ka.gdp_n = gdp_n;
    if (c.T > 0) {
        if ((st = make_map(&km, k, Tm * gdp_n, c.HK, c.K, k_st, k_sh)) != LA_OK) return st;
        if ((st = make_map(&vm, v, Tm * gdp_n, c.HV, c.V, v_st, v_sh)) != LA_OK) return st;
        if (q) {
            if ((st = make_map(&qm, q, Tm, c.HK, c.K, q_st, q_sh, qrows)) != LA_OK) return st;
        } else {
            qm = km;
        }
        // o goes out by TMA stores when its layout allows (16-byte base and strides); otherwise
        // the kernel stores it element by element
        // (GDP: only when n divides 64, so that every full chunk holds 64 / n whole tokens)
        ka.o_tma = 0;
        if (ka.o && aligned(ka.o, 16) && ka.o_st % 8 == 0 && (c.HV == 1 || ka.o_sh % 8 == 0) &&
            la::kChunk % gdp_n == 0 && make_map(&om, ka.o, Tm, c.HV, c.V, ka.o_st, ka.o_sh, qrows) == LA_OK)
            ka.o_tma = 1;
    }
    cudaEvent_t ev0 = t_timing_start, ev1 = t_timing_stop;
    t_timing_start = t_timing_stop = nullptr;
    if (ev0 && cudaEventRecord(ev0, stream) != cudaSuccess) return LA_ERR_CUDA;
    if (split) {
        ChunkArgs kw = ka;
        kw.num_units = SL.items;  // the bound on (chunk, head) items
        const int kind = mode == la::kModeSummary ? la::kWySummary : mode == la::kModeGdp ? la::kWyGdp : la::kWyFwd;
        if (la::launch_wy_kernel(kw, qm, km, wm, kind, stream) != cudaSuccess) return LA_ERR_CUDA;
    }
    const int kmode = !split ? mode
                             : (mode == la::kModeSummary ? la::kModeSummarySplit
                                                         : mode == la::kModeGdp ? la::kModeGdpSplit : la::kModeFwdSplit);
    if (la::launch_chunk_kernel(ka, qm, km, vm, om, wm, kmode, stream) != cudaSuccess) return LA_ERR_CUDA;
    if (ev1 && cudaEventRecord(ev1, stream) != cudaSuccess) return LA_ERR_CUDA;
    return LA_OK;
}

// ---------------------------------------------------------------------------
// Device-resident scratch for callers that cannot allocate device memory.
//
// Some callers are not allowed to call cudaMalloc at all: code running under
// an allocator that owns every byte of device memory (a framework's caching
// pool, a serving process that reserved all memory up front), or code that must
// not allocate after start-up.  gdn_fwd_static_workspace serves them with this
// file-scope array instead of a caller workspace or the library's lazily
// allocated one.  It lives in every GPU that loads the library until the
// process exits.  Its size covers the prologue's tables for up to
// kStaticMaxSeqs sequences (the unit order and the checkpoint row offsets).
// ---------------------------------------------------------------------------
constexpr int32_t kStaticMaxSeqs = 8192;
constexpr size_t kStaticScratchBytes = 98560;  // == la::ws_layout(kStaticMaxSeqs).total
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_static_mutex;
void* g_static_scratch_addr[128] = {};

// The host-side name g_static_scratch is only a stand-in, so the array's device
// address is looked up once per device, with that device current.
la_status static_scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return LA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_static_mutex);
    if (!g_static_scratch_addr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) return LA_ERR_CUDA;
        g_static_scratch_addr[dev] = ptr;
    }
    *out = g_static_scratch_addr[dev];
    return LA_OK;
}

}  // namespace

namespace {
la_status gdp_fwd(const la_gdn_fwd_params* p, void* stream);  // Gated DeltaProduct, below
la_status fwd_impl(const la_gdn_fwd_params* p, void* stream, int32_t gdp_n);
}  // namespace

extern "C" {

la_status gdn_fwd(const la_gdn_fwd_params* p, void* stream) {
    if (!p) return LA_ERR_INVALID_ARG;
    if (p->num_householder > 1) return gdp_fwd(p, stream);
    if (p->num_householder < 0) return LA_ERR_INVALID_ARG;
    return fwd_impl(p, stream, 1);
}

}  // extern "C"

namespace {
// The forward (gdp_n = 1) or Gated DeltaProduct natively on the update timeline (2 <= gdp_n <= 64).
la_status fwd_impl(const la_gdn_fwd_params* p, void* stream, int32_t gdp_n) {
    Common c{p->T, p->N, p->HK, p->HV, p->K, p->V, p->cu_seqlens, p->cu_seqlens_bits, p->g, p->beta,
             p->beta_bf16 ? 2 : 4};
    la_status st = check_common(c);
    if (st != LA_OK) return st;
    if (p->T > 0) {
        if ((st = check_tma_operand(p->q, p->q_stride_t, p->q_stride_h, p->HK)) != LA_OK) return st;
        if ((st = check_tma_operand(p->k, p->k_stride_t, p->k_stride_h, p->HK)) != LA_OK) return st;
        if ((st = check_tma_operand(p->v, p->v_stride_t, p->v_stride_h, p->HV)) != LA_OK) return st;
        if (!p->o || !aligned(p->o, 2) || p->o_stride_t <= 0 || (p->HV > 1 && p->o_stride_h <= 0))
            return LA_ERR_INVALID_ARG;
    }
    if (p->initial_state) {
        if (p->initial_state_dtype != LA_DTYPE_F32 && p->initial_state_dtype != LA_DTYPE_BF16) return LA_ERR_UNSUPPORTED;
        if (!aligned(p->initial_state, p->initial_state_dtype == LA_DTYPE_F32 ? 4 : 2)) return LA_ERR_INVALID_ARG;
    }
    if (p->final_state && !aligned(p->final_state, 4)) return LA_ERR_INVALID_ARG;
    if (p->checkpoints) {
        // a multiple of the chunk on the timeline the kernel walks (GDP: n update rows per token)
        if (p->checkpoint_every_n <= 0 || (p->checkpoint_every_n * gdp_n) % la::kChunk != 0) return LA_ERR_INVALID_ARG;
        if (p->checkpoint_dtype != LA_DTYPE_F32 && p->checkpoint_dtype != LA_DTYPE_BF16) return LA_ERR_UNSUPPORTED;
        if (!aligned(p->checkpoints, p->checkpoint_dtype == LA_DTYPE_F32 ? 4 : 2)) return LA_ERR_INVALID_ARG;
    }
    if (gdp_n > 1 && p->T > 0 && p->T * gdp_n >= (int64_t(1) << 31) - 64) return LA_ERR_UNSUPPORTED;
    ChunkArgs ka;
    std::memset(&ka, 0, sizeof(ka));
    ka.g_st = p->g_stride_t;
    ka.g_sh = p->g_stride_h;
    ka.b_st = p->beta_stride_t;
    ka.b_sh = p->beta_stride_h;
    ka.scale = p->scale > 0.f ? p->scale : 1.0f / std::sqrt(static_cast<float>(p->K));
    ka.l2norm = p->use_qk_l2norm != 0;
    ka.s0 = p->initial_state;
    ka.s0_bf16 = p->initial_state_dtype == LA_DTYPE_BF16;
    ka.o = static_cast<uint16_t*>(p->o);
    ka.o_st = p->o_stride_t;
    ka.o_sh = p->o_stride_h;
    ka.final_state = p->final_state;
    ka.ckpt = p->checkpoints;
    ka.ckpt_bf16 = p->checkpoint_dtype == LA_DTYPE_BF16;
    ka.ckpt_n = p->checkpoints ? p->checkpoint_every_n * gdp_n : 0;  // on the update timeline
    ka.transition = nullptr;
    ka.tiles_per_head = 1;
    if ((st = set_transforms(ka, p->gate_mode, p->a_log, p->dt_bias, p->gate_lower_bound, p->beta_sigmoid,
                             p->beta_bf16)) != LA_OK)
        return st;
    if (p->state_indices) {
        // state pool: the end states go back into initial_state in place
        if (!p->initial_state || p->final_state || p->checkpoints || p->state_pool_size <= 0 ||
            !aligned(p->state_indices, 4))
            return LA_ERR_INVALID_ARG;
        ka.state_idx = p->state_indices;
        ka.pool_size = p->state_pool_size;
        ka.final_state = static_cast<float*>(const_cast<void*>(p->initial_state));
        ka.final_bf16 = p->initial_state_dtype == LA_DTYPE_BF16;
    }
    return run(c, ka, p->q, p->q_stride_t, p->q_stride_h, p->k, p->k_stride_t, p->k_stride_h, p->v, p->v_stride_t,
               p->v_stride_h, p->checkpoints ? p->checkpoint_every_n : 0, p->workspace, p->workspace_bytes,
               p->status, gdp_n > 1 ? la::kModeGdp : la::kModeFwd, static_cast<cudaStream_t>(stream), gdp_n);
}
}  // namespace

extern "C" {

la_status gdn_decode(const la_gdn_decode_params* p, void* stream) {
    if (!p) return LA_ERR_INVALID_ARG;
    if (p->N < 0 || p->HK <= 0 || p->HV <= 0) return LA_ERR_INVALID_ARG;
    if ((p->K != 64 && p->K != 128) || (p->V != 64 && p->V != 128)) return LA_ERR_UNSUPPORTED;
    if (p->HV % p->HK != 0) return LA_ERR_UNSUPPORTED;
    if (p->state_dtype != LA_DTYPE_F32 && p->state_dtype != LA_DTYPE_BF16) return LA_ERR_UNSUPPORTED;
    if (!p->state_pool || !aligned(p->state_pool, 16) || p->state_pool_size <= 0) return LA_ERR_INVALID_ARG;
    if (!p->state_indices && p->state_pool_size < p->N) return LA_ERR_INVALID_ARG;
    if (p->state_indices && !aligned(p->state_indices, 4)) return LA_ERR_INVALID_ARG;
    if (static_cast<int64_t>(p->N) * p->HV >= (int64_t(1) << 31)) return LA_ERR_UNSUPPORTED;
    if (p->N > 0) {
        if (!p->q || !p->k || !p->v || !p->o || !p->g || !p->beta) return LA_ERR_INVALID_ARG;
        if (!aligned(p->q, 2) || !aligned(p->k, 2) || !aligned(p->v, 2) || !aligned(p->o, 2) || !aligned(p->g, 4) ||
            !aligned(p->beta, p->beta_bf16 ? 2 : 4))
            return LA_ERR_INVALID_ARG;
    }
    ChunkArgs tr;  // transform fields validated the same way as for gdn_fwd
    std::memset(&tr, 0, sizeof(tr));
    la_status st = set_transforms(tr, p->gate_mode, p->a_log, p->dt_bias, p->gate_lower_bound, p->beta_sigmoid,
                                  p->beta_bf16);
    if (st != LA_OK) return st;
    la::DecodeArgs d;
    std::memset(&d, 0, sizeof(d));
    d.q = static_cast<const uint16_t*>(p->q); d.q_sn = p->q_stride_n; d.q_sh = p->q_stride_h;
    d.k = static_cast<const uint16_t*>(p->k); d.k_sn = p->k_stride_n; d.k_sh = p->k_stride_h;
    d.v = static_cast<const uint16_t*>(p->v); d.v_sn = p->v_stride_n; d.v_sh = p->v_stride_h;
    d.g = p->g; d.g_sn = p->g_stride_n; d.g_sh = p->g_stride_h;
    d.beta = p->beta; d.b_sn = p->beta_stride_n; d.b_sh = p->beta_stride_h;
    d.N = p->N; d.HK = p->HK; d.HV = p->HV; d.K = p->K; d.V = p->V; d.group = p->HV / p->HK;
    d.scale = p->scale > 0.f ? p->scale : 1.0f / std::sqrt(static_cast<float>(p->K));
    d.l2norm = p->use_qk_l2norm != 0;
    d.pool = p->state_pool; d.pool_bf16 = p->state_dtype == LA_DTYPE_BF16; d.pool_size = p->state_pool_size;
    d.idx = p->state_indices;
    d.o = static_cast<uint16_t*>(p->o); d.o_sn = p->o_stride_n; d.o_sh = p->o_stride_h;
    d.status = p->status;
    d.gate_mode = tr.gate_mode; d.a_log = tr.a_log; d.dt_bias = tr.dt_bias; d.gate_lb = tr.gate_lb;
    d.beta_sigmoid = tr.beta_sigmoid; d.beta_bf16 = tr.beta_bf16;
    cudaEvent_t ev0 = t_timing_start, ev1 = t_timing_stop;
    t_timing_start = t_timing_stop = nullptr;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (ev0 && cudaEventRecord(ev0, s) != cudaSuccess) return LA_ERR_CUDA;
    if (la::launch_decode(d, s) != cudaSuccess) return LA_ERR_CUDA;
    if (ev1 && cudaEventRecord(ev1, s) != cudaSuccess) return LA_ERR_CUDA;
    return LA_OK;
}

}  // extern "C"

namespace {
struct GdpLayout {
    size_t pro, qe, ge, cue, oe, total;
};
GdpLayout gdp_layout(int64_t T, int32_t N, int32_t HK, int32_t HV, int32_t K, int32_t V, int32_t n) {
    GdpLayout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += (bytes + 255) & ~size_t(255);
        return at;
    };
    // the forward on the timeline (T n rows) gets room for its two-pass schedule
    L.pro = take(la::split_layout(T * n, N, HV).total);
    L.qe = take(static_cast<size_t>(T) * n * HK * K * 2);
    L.ge = take(static_cast<size_t>(T) * n * HV * sizeof(float));
    L.cue = take(static_cast<size_t>(N + 1) * sizeof(int64_t));
    L.oe = take(static_cast<size_t>(T) * n * HV * V * 2);
    L.total = off;
    return L;
}
}  // namespace

extern "C" size_t la_gdp_workspace_bytes(int64_t T, int32_t N, int32_t HK, int32_t HV, int32_t K, int32_t V,
                                         int32_t n) {
    if (T < 0 || N < 0 || HK <= 0 || HV <= 0 || n < 1) return 0;
    if (n == 1) return la::ws_layout(N).total;
    // n <= 64 runs natively on the update timeline: the two-pass workspace of that timeline
    if (n <= la::kChunk) return la::split_layout(T * n, N, HV).total;
    return gdp_layout(T, N, HK, HV, K, V, n).total;
}

namespace {
// GDP: build the update timeline (query, gate, boundaries), run the GDN path on it, gather the
// per-token outputs.
la_status gdp_fwd(const la_gdn_fwd_params* p, void* stream) {
    const int32_t n = p->num_householder;
    // n <= 64: natively on the update timeline (q, g, o read and written on the token timeline
    // by the chunk kernel); larger n: the timeline's query, gate and output rows are
    // materialised below and the plain forward runs on it
    if (n <= la::kChunk) return fwd_impl(p, stream, n);
    if (p->N < 0 || p->HK <= 0 || p->HV <= 0 || p->T < 0) return LA_ERR_INVALID_ARG;
    if ((p->K != 64 && p->K != 128) || (p->V != 64 && p->V != 128)) return LA_ERR_UNSUPPORTED;
    if (p->HV % p->HK != 0) return LA_ERR_UNSUPPORTED;
    if (p->T * n >= (int64_t(1) << 31) - 64) return LA_ERR_UNSUPPORTED;
    if (p->cu_seqlens_bits != 32 && p->cu_seqlens_bits != 64) return LA_ERR_INVALID_ARG;
    if (!p->cu_seqlens) return LA_ERR_INVALID_ARG;
    if (p->T > 0) {
        if (!p->q || !aligned(p->q, 16) || p->q_stride_t % 8 != 0 || (p->HK > 1 && p->q_stride_h % 8 != 0))
            return LA_ERR_INVALID_ARG;
        if (!p->g || !aligned(p->g, 4) || !p->o || !aligned(p->o, 2)) return LA_ERR_INVALID_ARG;
    }
    const GdpLayout GL = gdp_layout(p->T, p->N, p->HK, p->HV, p->K, p->V, n);
    void* ws = p->workspace;
    la_status st;
    if (ws) {
        if (p->workspace_bytes < GL.total || !aligned(ws, 256)) return LA_ERR_WORKSPACE;
    } else if ((st = internal_workspace(GL.total, static_cast<cudaStream_t>(stream), &ws)) != LA_OK) {
        return st;
    }
    uint8_t* wb = static_cast<uint8_t*>(ws);
    ChunkArgs tr;  // the gate transform is applied while the gate rows are built
    std::memset(&tr, 0, sizeof(tr));
    if ((st = set_transforms(tr, p->gate_mode, p->a_log, p->dt_bias, p->gate_lower_bound, p->beta_sigmoid,
                             p->beta_bf16)) != LA_OK)
        return st;
    la::GdpArgs g;
    std::memset(&g, 0, sizeof(g));
    g.T = p->T; g.N = p->N; g.HK = p->HK; g.HO = p->HV; g.K = p->K; g.V = p->V; g.n = n;
    g.q = static_cast<const uint16_t*>(p->q); g.q_st = p->q_stride_t; g.q_sh = p->q_stride_h;
    g.g = p->g; g.g_st = p->g_stride_t; g.g_sh = p->g_stride_h;
    g.cu = p->cu_seqlens; g.cu64 = p->cu_seqlens_bits == 64;
    g.gate_mode = tr.gate_mode; g.a_log = tr.a_log; g.dt_bias = tr.dt_bias; g.gate_lb = tr.gate_lb;
    g.qe = reinterpret_cast<uint16_t*>(wb + GL.qe);
    g.ge = reinterpret_cast<float*>(wb + GL.ge);
    g.cue = reinterpret_cast<int64_t*>(wb + GL.cue);
    g.oe = reinterpret_cast<const uint16_t*>(wb + GL.oe);
    g.o = static_cast<uint16_t*>(p->o); g.o_st = p->o_stride_t; g.o_sh = p->o_stride_h;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (la::launch_gdp_expand(g, s) != cudaSuccess) return LA_ERR_CUDA;
    la_gdn_fwd_params f = *p;
    f.num_householder = 1;
    f.q = g.qe; f.q_stride_t = static_cast<int64_t>(p->HK) * p->K; f.q_stride_h = p->K;
    f.g = g.ge; f.g_stride_t = p->HV; f.g_stride_h = 1;
    f.gate_mode = LA_GATE_LOG; f.a_log = nullptr; f.dt_bias = nullptr;
    f.cu_seqlens = g.cue; f.cu_seqlens_bits = 64;
    f.T = p->T * n;
    f.o = wb + GL.oe; f.o_stride_t = static_cast<int64_t>(p->HV) * p->V; f.o_stride_h = p->V;
    f.checkpoint_every_n = p->checkpoints ? p->checkpoint_every_n * n : 0;
    f.workspace = wb + GL.pro; f.workspace_bytes = la::split_layout(p->T * n, p->N, p->HV).total;
    if ((st = gdn_fwd(&f, stream)) != LA_OK) return st;
    if (la::launch_gdp_gather(g, s) != cudaSuccess) return LA_ERR_CUDA;
    return LA_OK;
}

// How the backward gets the fp32 states entering every chunk.
enum BwdCkpt : int {
    kCkNone = 0,     // regenerated by a forward pass over the batch
    kCkDirect = 1,   // given: fp32 rows every 64 tokens
    kCkWiden = 2,    // given: bf16 rows every 64 tokens, widened to fp32
    kCkSegments = 3  // given: rows every n > 64 tokens; the forward over the n-token segments
};
int bwd_ckpt_mode(bool given, int64_t n, bool bf16) {
    if (!given) return kCkNone;
    if (n == 0 || n == la::kChunk) return bf16 ? kCkWiden : kCkDirect;
    return kCkSegments;
}
// the segments of a batch cut at multiples of n: at most ceil(T / n) + N of them
int64_t max_segments(int64_t T, int32_t N, int64_t n) { return (T + n - 1) / n + N; }

struct BwdLayout {
    size_t pro, ck, o, ds, gh, gp, pro_n, pro_seg, cu_seg, s0_seg, total;
    // the tensor-core path (K = V = 128) after the rest: the split layout's prologue area, chunk
    // numbering and WY records, the gradient leaving every (chunk, head), per-item gate sums
    size_t tc_split, tc_ds, tc_tlo, tc_gp, tc_carry, tc_flags, total_tc;
};
size_t up256(size_t x) { return (x + 255) & ~size_t(255); }
BwdLayout bwd_layout(int64_t T, int32_t N, int32_t HK, int32_t HV, int32_t K, int32_t V, int mode, int64_t n = 0) {
    BwdLayout L{};
    size_t off = up256(la::ws_layout(N).total);
    const size_t rows = static_cast<size_t>((T + la::kChunk - 1) / la::kChunk + N);  // >= sum ceil(L_i / 64)
    L.pro = 0;
    L.ck = off;
    if (mode != kCkDirect) off += up256(rows * HV * K * V * sizeof(float));
    L.o = off;
    if (mode == kCkNone || mode == kCkSegments) off += up256(static_cast<size_t>(T) * HV * V * 2);
    L.ds = off;
    off += up256(static_cast<size_t>(N) * HV * K * V * sizeof(float));
    L.gh = off;
    if (HV != HK) off += up256(2 * static_cast<size_t>(T) * HV * K * sizeof(float));
    L.gp = off;  // per (sequence, head, chunk range) sums for the softplus gate's parameter gradients
    off += up256(2 * static_cast<size_t>(N) * HV * la::kBwdPieces * sizeof(float));
    if (mode == kCkSegments) {
        // the cadence-n row offsets, the segments' own prologue area, boundaries and start states
        const int64_t S = max_segments(T, N, n);
        L.pro_n = off;
        off += up256(la::ws_layout(N).total);
        L.pro_seg = off;
        off += up256(la::ws_layout(static_cast<int32_t>(S)).total);
        L.cu_seg = off;
        off += up256(static_cast<size_t>(S + 1) * sizeof(int64_t));
        L.s0_seg = off;
        off += up256(static_cast<size_t>(S) * HV * K * V * sizeof(float));
    }
    L.total = off;
    const la::SplitLayout GL = la::split_layout(T, N, HV);
    L.tc_split = off;
    off += up256(GL.total);
    L.tc_ds = off;
    off += up256(static_cast<size_t>(GL.items) * 65536);
    L.tc_tlo = off;
    off += up256(static_cast<size_t>(GL.items) * la::kWyTileBytes);
    L.tc_gp = off;
    off += up256(2 * static_cast<size_t>(HV) * static_cast<size_t>(GL.chunks) * sizeof(float));
    L.tc_carry = off;  // the state-gradient pass's range hand-off and its flags
    off += up256(static_cast<size_t>(N) * HV * K * V * sizeof(float));
    L.tc_flags = off;
    off += up256(static_cast<size_t>(N) * HV * sizeof(int32_t));
    L.total_tc = off;
    return L;
}
// the full backward runs on the tensor cores for K = V = 128 (else the tile kernel)
bool bwd_tc_shape(int32_t K, int32_t V) { return K == 128 && V == 128; }
// gdn_summary_bwd: the prologue's area, then the carried state gradient of every (sequence, head).
struct SumBwdLayout {
    size_t pro, ds, total;
};
SumBwdLayout sum_bwd_layout(int32_t N, int32_t HV, int32_t K, int32_t V) {
    SumBwdLayout L{};
    L.pro = 0;
    L.ds = up256(la::ws_layout(N).total);
    L.total = L.ds + up256(static_cast<size_t>(N) * HV * K * V * sizeof(float));
    return L;
}
}  // namespace

extern "C" {

size_t la_gdn_summary_bwd_workspace_bytes(int32_t N, int32_t HV, int32_t K, int32_t V) {
    if (N < 0 || HV <= 0 || K <= 0 || V <= 0) return 0;
    return sum_bwd_layout(N, HV, K, V).total;
}

size_t la_gdn_bwd_workspace_bytes(int64_t T, int32_t N, int32_t HK, int32_t HV, int32_t K, int32_t V,
                                  int32_t checkpoints_given) {
    if (T < 0 || N < 0 || HK <= 0 || HV <= 0) return 0;
    const BwdLayout L = bwd_layout(T, N, HK, HV, K, V, checkpoints_given != 0 ? kCkDirect : kCkNone);
    return bwd_tc_shape(K, V) ? L.total_tc : L.total;
}

size_t la_gdn_bwd_workspace_bytes_ckpt(int64_t T, int32_t N, int32_t HK, int32_t HV, int32_t K, int32_t V,
                                       int64_t checkpoint_every_n, int32_t checkpoint_bf16) {
    if (T < 0 || N < 0 || HK <= 0 || HV <= 0 || checkpoint_every_n < 0 || checkpoint_every_n % la::kChunk != 0)
        return 0;
    const int mode = bwd_ckpt_mode(checkpoint_every_n > 0, checkpoint_every_n, checkpoint_bf16 != 0);
    const BwdLayout L = bwd_layout(T, N, HK, HV, K, V, mode, checkpoint_every_n);
    return bwd_tc_shape(K, V) ? L.total_tc : L.total;
}

}  // extern "C"

namespace {
// gdn_bwd on the tensor cores (K = V = 128), once the states entering every chunk are in
// b.ckpt: the prologue (chunk numbering), the forward's WY pass over every (chunk, head), the
// state-gradient pass (the gradient leaving every chunk into the workspace, d_initial_state),
// the chunk-parallel gradient pass, then the grouped-head and gate-parameter sums.
la_status bwd_tensor_path(const la_gdn_bwd_params* p, const BwdLayout& BL, uint8_t* wb, la::BwdArgs b,
                          cudaStream_t s) {
    la_status st;
    const la::SplitLayout GL = la::split_layout(p->T, p->N, p->HV);
    uint8_t* gw = wb + BL.tc_split;
    const la::WorkspaceLayout PL = la::ws_layout(p->N);
    PrologueArgs pa;
    pa.cu = p->cu_seqlens;
    pa.chunk_off = reinterpret_cast<int64_t*>(gw + GL.chunk_off);
    pa.chunk_seq = reinterpret_cast<int32_t*>(gw + GL.chunk_seq);
    pa.chunk_rows = 1;
    pa.cu64 = p->cu_seqlens_bits == 64;
    pa.T = p->T;
    pa.N = p->N;
    pa.ckpt_n = 0;
    pa.hdr = reinterpret_cast<la::WsHeader*>(gw);
    pa.order = reinterpret_cast<int32_t*>(gw + PL.order);
    pa.ckpt_off = reinterpret_cast<int64_t*>(gw + PL.ckpt_off);
    pa.keys = reinterpret_cast<uint64_t*>(gw + PL.keys);
    pa.user_status = p->status;
    if (la::launch_prologue(pa, s) != cudaSuccess) return LA_ERR_CUDA;

    ChunkArgs ka;
    std::memset(&ka, 0, sizeof(ka));
    if ((st = set_transforms(ka, p->gate_mode, p->a_log, p->dt_bias, p->gate_lower_bound, p->beta_sigmoid,
                             p->beta_bf16)) != LA_OK)
        return st;
    ka.g = p->g;
    ka.g_st = p->g_stride_t;
    ka.g_sh = p->g_stride_h;
    ka.beta = p->beta;
    ka.b_st = p->beta_stride_t;
    ka.b_sh = p->beta_stride_h;
    ka.cu = p->cu_seqlens;
    ka.cu64 = p->cu_seqlens_bits == 64;
    ka.T = p->T;
    ka.N = p->N;
    ka.HK = p->HK;
    ka.HV = p->HV;
    ka.K = p->K;
    ka.V = p->V;
    ka.group = p->HV / p->HK;
    ka.scale = b.scale;
    ka.l2norm = p->use_qk_l2norm != 0;
    ka.s0 = p->d_final_state;
    ka.final_state = p->d_initial_state;
    ka.tiles_per_head = 1;
    ka.num_units = static_cast<int64_t>(p->N) * p->HV;
    ka.hdr = pa.hdr;
    ka.order = pa.order;
    ka.ckpt_off = pa.ckpt_off;
    ka.chunk_off = pa.chunk_off;
    ka.chunk_seq = pa.chunk_seq;
    ka.wy = gw + GL.wy;
    ka.ds_chunks = wb + BL.tc_ds;
    ka.grad_carry = reinterpret_cast<float*>(wb + BL.tc_carry);
    ka.grad_flags = reinterpret_cast<int32_t*>(wb + BL.tc_flags);
    ka.user_status = p->status;
    ka.wait_budget_ns = kWaitBudgetNs;
    ka.gdp_n = 1;
    if (const uint64_t wb_ns = g_test_wait_budget_ns.load(std::memory_order_relaxed)) ka.wait_budget_ns = wb_ns;

    CUtensorMap qm, km, dom, wm;
    if ((st = make_map(&km, p->k, p->T, p->HK, p->K, p->k_stride_t, p->k_stride_h)) != LA_OK) return st;
    if ((st = make_map(&qm, p->q, p->T, p->HK, p->K, p->q_stride_t, p->q_stride_h)) != LA_OK) return st;
    if ((st = make_map(&dom, p->d_o, p->T, p->HV, p->V, p->d_o_stride_t, p->d_o_stride_h)) != LA_OK) return st;
    if ((st = make_map(&wm, ka.wy, 136, GL.items, 64, 64, static_cast<int64_t>(la::kWyRecordBytes / 2))) != LA_OK)
        return st;
    // per-item gate-parameter sums: slot (head, chunk) over the chunk bound, unused slots zero
    b.N = 1;
    b.pieces = static_cast<int32_t>(GL.chunks);
    if (b.gpart) {
        b.gpart = reinterpret_cast<float*>(wb + BL.tc_gp);
        if (cudaMemsetAsync(b.gpart, 0, 2 * static_cast<size_t>(p->HV) * GL.chunks * sizeof(float), s) != cudaSuccess)
            return LA_ERR_CUDA;
    }
    ka.wy_tlo = wb + BL.tc_tlo;
    // full chunks of dq, dk, dv leave by TMA when the output rows allow it
    b.out_tma = b.vec_out && aligned(p->dv, 16) && p->dv_stride_t % 8 == 0 && (p->HV == 1 || p->dv_stride_h % 8 == 0);
    CUtensorMap dkm, dqm, dvm;
    std::memset(&dkm, 0, sizeof(dkm));
    std::memset(&dqm, 0, sizeof(dqm));
    std::memset(&dvm, 0, sizeof(dvm));
    if (b.out_tma && (make_map(&dkm, p->dk, p->T, p->HK, p->K, p->dk_stride_t, p->dk_stride_h) != LA_OK ||
                      make_map(&dqm, p->dq, p->T, p->HK, p->K, p->dq_stride_t, p->dq_stride_h) != LA_OK ||
                      make_map(&dvm, p->dv, p->T, p->HV, p->V, p->dv_stride_t, p->dv_stride_h) != LA_OK))
        b.out_tma = 0;  // (per-thread stores then)
    ChunkArgs kw = ka;
    kw.num_units = GL.items;  // the bound on (chunk, head) items
    if (la::launch_wy_kernel(kw, qm, km, wm, la::kWyFwd, s) != cudaSuccess) return LA_ERR_CUDA;
    if (la::launch_grad(ka, qm, km, dom, wm, s) != cudaSuccess) return LA_ERR_CUDA;
    ChunkArgs kd = ka;
    kd.items = GL.items;
    // the failure-path test hook reaches the chunk pass only (its first tile wait runs out)
    kd.test_skip_tile_load = g_test_skip_tile_load.load(std::memory_order_relaxed) != 0;
    if (la::launch_dchunk(kd, b, qm, km, dom, wm, dkm, dqm, dvm, s) != cudaSuccess) return LA_ERR_CUDA;
    if (la::launch_bwd_finish(b, s) != cudaSuccess) return LA_ERR_CUDA;
    return LA_OK;
}
}  // namespace

extern "C" {

size_t la_gdn_bwd_workspace_bytes_min(int64_t T, int32_t N, int32_t HK, int32_t HV, int32_t K, int32_t V,
                                      int64_t checkpoint_every_n, int32_t checkpoint_bf16) {
    if (T < 0 || N < 0 || HK <= 0 || HV <= 0 || checkpoint_every_n < 0 || checkpoint_every_n % la::kChunk != 0)
        return 0;
    const int mode = bwd_ckpt_mode(checkpoint_every_n > 0, checkpoint_every_n, checkpoint_bf16 != 0);
    return bwd_layout(T, N, HK, HV, K, V, mode, checkpoint_every_n).total;
}

la_status gdn_bwd(const la_gdn_bwd_params* p, void* stream) {
    if (!p) return LA_ERR_INVALID_ARG;
    Common c{p->T, p->N, p->HK, p->HV, p->K, p->V, p->cu_seqlens, p->cu_seqlens_bits, p->g, p->beta,
             p->beta_bf16 ? 2 : 4};
    la_status st = check_common(c);
    if (st != LA_OK) return st;
    la::BwdArgs b;
    std::memset(&b, 0, sizeof(b));
    if ((st = set_bwd_transforms(b, p->gate_mode, p->a_log, p->dt_bias, p->gate_lower_bound, p->beta_sigmoid,
                                 p->beta_bf16)) != LA_OK)
        return st;
    if ((p->d_a_log && !aligned(p->d_a_log, 4)) || (p->d_dt_bias && !aligned(p->d_dt_bias, 4))) return LA_ERR_INVALID_ARG;
    if (p->T > 0) {
        if ((st = check_tma_operand(p->q, p->q_stride_t, p->q_stride_h, p->HK)) != LA_OK) return st;
        if ((st = check_tma_operand(p->k, p->k_stride_t, p->k_stride_h, p->HK)) != LA_OK) return st;
        if ((st = check_tma_operand(p->v, p->v_stride_t, p->v_stride_h, p->HV)) != LA_OK) return st;
        if (!p->d_o || !p->dq || !p->dk || !p->dv || !p->dg || !p->dbeta) return LA_ERR_INVALID_ARG;
        if (!aligned(p->d_o, 2) || !aligned(p->dq, 2) || !aligned(p->dk, 2) || !aligned(p->dv, 2) ||
            !aligned(p->dg, 4) || !aligned(p->dbeta, 4))
            return LA_ERR_INVALID_ARG;
    }
    if (p->initial_state) {
        if (p->initial_state_dtype != LA_DTYPE_F32 && p->initial_state_dtype != LA_DTYPE_BF16) return LA_ERR_UNSUPPORTED;
        if (!aligned(p->initial_state, p->initial_state_dtype == LA_DTYPE_F32 ? 4 : 2)) return LA_ERR_INVALID_ARG;
    }
    if (p->checkpoint_every_n < 0 || p->checkpoint_every_n % la::kChunk != 0) return LA_ERR_INVALID_ARG;
    const bool ck_bf16 = p->checkpoint_bf16 != 0;
    if (p->checkpoints && !aligned(p->checkpoints, ck_bf16 ? 2 : 4)) return LA_ERR_INVALID_ARG;
    if ((p->d_final_state && !aligned(p->d_final_state, 4)) || (p->d_initial_state && !aligned(p->d_initial_state, 4)))
        return LA_ERR_INVALID_ARG;
    const int mode = bwd_ckpt_mode(p->checkpoints != nullptr, p->checkpoint_every_n, ck_bf16);
    const int64_t ck_n = mode == kCkSegments ? p->checkpoint_every_n : la::kChunk;
    const BwdLayout BL = bwd_layout(p->T, p->N, p->HK, p->HV, p->K, p->V, mode, ck_n);
    // the tensor-core path when the shapes, the d_o operand (TMA) and the workspace allow it
    const la::SplitLayout GLb = la::split_layout(p->T, p->N, p->HV);
    bool tc = g_test_fwd_passes.load(std::memory_order_relaxed) != 1 && p->T > 0 && bwd_tc_shape(p->K, p->V) &&
              GLb.items < (int64_t(1) << 31) && aligned(p->d_o, 16) && p->d_o_stride_t % 8 == 0 &&
              (p->HV == 1 || p->d_o_stride_h % 8 == 0);
    void* ws = p->workspace;
    if (ws) {
        if (p->workspace_bytes < BL.total || !aligned(ws, 256)) return LA_ERR_WORKSPACE;
        tc = tc && p->workspace_bytes >= BL.total_tc;
    } else {
        if (tc && internal_workspace(BL.total_tc, static_cast<cudaStream_t>(stream), &ws) != LA_OK) {
            tc = false;
            ws = nullptr;
        }
        if (!ws && (st = internal_workspace(BL.total, static_cast<cudaStream_t>(stream), &ws)) != LA_OK) return st;
    }
    uint8_t* wb = static_cast<uint8_t*>(ws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const float* ck = static_cast<const float*>(p->checkpoints);
    const la::WorkspaceLayout PL = la::ws_layout(p->N);
    const int64_t row_elems = static_cast<int64_t>(p->HV) * p->K * p->V;
    const int64_t rows64 = (p->T + la::kChunk - 1) / la::kChunk + p->N;  // the regenerated rows' capacity
    // the forward over the batch (or over its segments), writing fp32 states every 64 tokens
    auto regen_fwd = [&](la_gdn_fwd_params& f) {
        std::memset(&f, 0, sizeof(f));
        f.q = p->q; f.q_stride_t = p->q_stride_t; f.q_stride_h = p->q_stride_h;
        f.k = p->k; f.k_stride_t = p->k_stride_t; f.k_stride_h = p->k_stride_h;
        f.v = p->v; f.v_stride_t = p->v_stride_t; f.v_stride_h = p->v_stride_h;
        f.g = p->g; f.g_stride_t = p->g_stride_t; f.g_stride_h = p->g_stride_h;
        f.beta = p->beta; f.beta_stride_t = p->beta_stride_t; f.beta_stride_h = p->beta_stride_h;
        f.cu_seqlens = p->cu_seqlens; f.cu_seqlens_bits = p->cu_seqlens_bits;
        f.T = p->T; f.N = p->N; f.HK = p->HK; f.HV = p->HV; f.K = p->K; f.V = p->V;
        f.scale = p->scale; f.use_qk_l2norm = p->use_qk_l2norm;
        f.initial_state = p->initial_state; f.initial_state_dtype = p->initial_state_dtype;
        f.gate_mode = p->gate_mode; f.a_log = p->a_log; f.dt_bias = p->dt_bias;
        f.gate_lower_bound = p->gate_lower_bound; f.beta_sigmoid = p->beta_sigmoid; f.beta_bf16 = p->beta_bf16;
        f.o = wb + BL.o; f.o_stride_t = static_cast<int64_t>(p->HV) * p->V; f.o_stride_h = p->V;
        f.checkpoints = wb + BL.ck; f.checkpoint_dtype = LA_DTYPE_F32; f.checkpoint_every_n = la::kChunk;
        f.workspace = wb + BL.pro; f.workspace_bytes = PL.total;
        f.status = p->status;
    };
    // a prologue over the batch: validation and the checkpoint-row offsets at cadence n
    auto prologue = [&](size_t area, int64_t n) {
        PrologueArgs pa;
        pa.cu = p->cu_seqlens;
        pa.chunk_off = nullptr;
        pa.chunk_rows = 1;
        pa.cu64 = p->cu_seqlens_bits == 64;
        pa.T = p->T;
        pa.N = p->N;
        pa.ckpt_n = n;
        pa.hdr = reinterpret_cast<la::WsHeader*>(wb + area);
        pa.order = reinterpret_cast<int32_t*>(wb + area + PL.order);
        pa.ckpt_off = reinterpret_cast<int64_t*>(wb + area + PL.ckpt_off);
        pa.keys = reinterpret_cast<uint64_t*>(wb + area + PL.keys);
        pa.user_status = p->status;
        return la::launch_prologue(pa, s) == cudaSuccess ? LA_OK : LA_ERR_CUDA;
    };
    if (mode == kCkNone) {
        // states entering every chunk: the forward with fp32 checkpoints every 64 tokens
        la_gdn_fwd_params f;
        regen_fwd(f);
        if ((st = gdn_fwd(&f, stream)) != LA_OK) return st;
        ck = reinterpret_cast<const float*>(wb + BL.ck);
    } else if (mode == kCkDirect) {
        // only the prologue: validation and the chunk-row offsets of the caller's checkpoints (the
        // tensor-core schedule runs its own, which also numbers the chunks)
        tc = tc && aligned(ck, 16);
        if (!tc && (st = prologue(BL.pro, la::kChunk)) != LA_OK) return st;
    } else if (mode == kCkWiden) {
        // bf16 rows at the chunk cadence: widened to fp32
        if ((st = prologue(BL.pro, la::kChunk)) != LA_OK) return st;
        la::CkptArgs ca;
        std::memset(&ca, 0, sizeof(ca));
        ca.src = p->checkpoints;
        ca.src_bf16 = 1;
        ca.row_elems = row_elems;
        ca.hdr = reinterpret_cast<const la::WsHeader*>(wb + BL.pro);
        ca.max_rows = rows64;
        ca.dst = reinterpret_cast<float*>(wb + BL.ck);
        if (la::launch_ckpt_widen(ca, s) != cudaSuccess) return LA_ERR_CUDA;
        ck = reinterpret_cast<const float*>(wb + BL.ck);
    } else {
        // rows every n > 64 tokens: the forward over the n-token segments, each from its row,
        // writes the states entering every chunk in the order the backward reads them
        if ((st = prologue(BL.pro_n, ck_n)) != LA_OK) return st;
        const int64_t S = max_segments(p->T, p->N, ck_n);
        la::CkptArgs ca;
        std::memset(&ca, 0, sizeof(ca));
        ca.src = p->checkpoints;
        ca.src_bf16 = ck_bf16;
        ca.row_elems = row_elems;
        ca.hdr = reinterpret_cast<const la::WsHeader*>(wb + BL.pro_n);
        ca.cu = p->cu_seqlens;
        ca.cu64 = p->cu_seqlens_bits == 64;
        ca.N = p->N;
        ca.T = p->T;
        ca.n = ck_n;
        ca.ckpt_off_n = reinterpret_cast<const int64_t*>(wb + BL.pro_n + PL.ckpt_off);
        ca.cu_seg = reinterpret_cast<int64_t*>(wb + BL.cu_seg);
        ca.s0_seg = reinterpret_cast<float*>(wb + BL.s0_seg);
        ca.max_seg = S;
        if (la::launch_ckpt_segments(ca, s) != cudaSuccess) return LA_ERR_CUDA;
        la_gdn_fwd_params f;
        regen_fwd(f);
        f.cu_seqlens = wb + BL.cu_seg; f.cu_seqlens_bits = 64;
        f.N = static_cast<int32_t>(S);
        f.initial_state = wb + BL.s0_seg; f.initial_state_dtype = LA_DTYPE_F32;
        f.workspace = wb + BL.pro_seg; f.workspace_bytes = la::ws_layout(static_cast<int32_t>(S)).total;
        if ((st = gdn_fwd(&f, stream)) != LA_OK) return st;
        // the backward's own chunk-row offsets over the batch
        if ((st = prologue(BL.pro, la::kChunk)) != LA_OK) return st;
        ck = reinterpret_cast<const float*>(wb + BL.ck);
    }
    b.q = static_cast<const uint16_t*>(p->q); b.q_st = p->q_stride_t; b.q_sh = p->q_stride_h;
    b.k = static_cast<const uint16_t*>(p->k); b.k_st = p->k_stride_t; b.k_sh = p->k_stride_h;
    b.v = static_cast<const uint16_t*>(p->v); b.v_st = p->v_stride_t; b.v_sh = p->v_stride_h;
    b.g = p->g; b.g_st = p->g_stride_t; b.g_sh = p->g_stride_h;
    b.beta = p->beta; b.b_st = p->beta_stride_t; b.b_sh = p->beta_stride_h;
    b.cu = p->cu_seqlens; b.cu64 = p->cu_seqlens_bits == 64;
    b.T = p->T; b.N = p->N; b.HK = p->HK; b.HV = p->HV; b.K = p->K; b.V = p->V; b.group = p->HV / p->HK;
    b.scale = p->scale > 0.f ? p->scale : 1.0f / std::sqrt(static_cast<float>(p->K));
    b.l2norm = p->use_qk_l2norm != 0;
    b.dout = static_cast<const uint16_t*>(p->d_o); b.do_st = p->d_o_stride_t; b.do_sh = p->d_o_stride_h;
    b.dfinal = p->d_final_state;
    b.ckpt = ck;
    b.ckpt_off = reinterpret_cast<const int64_t*>(wb + BL.pro + PL.ckpt_off);
    b.hdr = reinterpret_cast<const la::WsHeader*>(wb + BL.pro);
    b.dS_work = reinterpret_cast<float*>(wb + BL.ds);
    b.dq = static_cast<uint16_t*>(p->dq); b.dq_st = p->dq_stride_t; b.dq_sh = p->dq_stride_h;
    b.dk = static_cast<uint16_t*>(p->dk); b.dk_st = p->dk_stride_t; b.dk_sh = p->dk_stride_h;
    b.dv = static_cast<uint16_t*>(p->dv); b.dv_st = p->dv_stride_t; b.dv_sh = p->dv_stride_h;
    b.dg = p->dg; b.dg_st = p->dg_stride_t; b.dg_sh = p->dg_stride_h;
    b.dbeta = p->dbeta; b.db_st = p->dbeta_stride_t; b.db_sh = p->dbeta_stride_h;
    b.ds0 = p->d_initial_state;
    b.vec_out = aligned(p->dq, 16) && aligned(p->dk, 16) && p->dq_stride_t % 8 == 0 && p->dk_stride_t % 8 == 0 &&
                (p->HK == 1 || (p->dq_stride_h % 8 == 0 && p->dk_stride_h % 8 == 0));
    b.vo_async = aligned(p->v, 4) && aligned(p->d_o, 4) && p->v_stride_t % 2 == 0 && p->d_o_stride_t % 2 == 0 &&
                 (p->HV == 1 || (p->v_stride_h % 2 == 0 && p->d_o_stride_h % 2 == 0));
    if (p->HV != p->HK) {
        b.dqh = reinterpret_cast<float*>(wb + BL.gh);
        b.dkh = b.dqh + static_cast<size_t>(p->T) * p->HV * p->K;
    }
    if (b.gate_mode == LA_GATE_SOFTPLUS && (p->d_a_log || p->d_dt_bias)) {
        b.gpart = reinterpret_cast<float*>(wb + BL.gp);
        b.d_a_log = p->d_a_log;
        b.d_dt_bias = p->d_dt_bias;
    }
    tc = tc && aligned(ck, 16);  // the states arrive by bulk copy
    cudaEvent_t ev0 = t_timing_start, ev1 = t_timing_stop;
    t_timing_start = t_timing_stop = nullptr;
    if (ev0 && cudaEventRecord(ev0, s) != cudaSuccess) return LA_ERR_CUDA;
    if (tc) {
        if ((st = bwd_tensor_path(p, BL, wb, b, s)) != LA_OK) return st;
    } else if (la::launch_bwd(b, s) != cudaSuccess) {
        return LA_ERR_CUDA;
    }
    if (ev1 && cudaEventRecord(ev1, s) != cudaSuccess) return LA_ERR_CUDA;
    return LA_OK;
}

namespace {
// gdn_summary_bwd on the tensor cores: the prologue (validation, longest-first order, chunk
// numbering), the forward's WY pass over every (chunk, head), and the state-gradient pass.
la_status summary_bwd_two_pass(const la_gdn_summary_bwd_params* p, const la::SplitLayout& GL, uint8_t* wb,
                               cudaStream_t s) {
    la_status st;
    const la::WorkspaceLayout PL = la::ws_layout(p->N);
    PrologueArgs pa;
    pa.cu = p->cu_seqlens;
    pa.chunk_off = reinterpret_cast<int64_t*>(wb + GL.chunk_off);
    pa.chunk_seq = reinterpret_cast<int32_t*>(wb + GL.chunk_seq);
    pa.chunk_rows = 1;
    pa.cu64 = p->cu_seqlens_bits == 64;
    pa.T = p->T;
    pa.N = p->N;
    pa.ckpt_n = 0;
    pa.hdr = reinterpret_cast<la::WsHeader*>(wb);
    pa.order = reinterpret_cast<int32_t*>(wb + PL.order);
    pa.ckpt_off = reinterpret_cast<int64_t*>(wb + PL.ckpt_off);
    pa.keys = reinterpret_cast<uint64_t*>(wb + PL.keys);
    pa.user_status = p->status;
    if (la::launch_prologue(pa, s) != cudaSuccess) return LA_ERR_CUDA;

    ChunkArgs ka;
    std::memset(&ka, 0, sizeof(ka));
    if ((st = set_transforms(ka, p->gate_mode, p->a_log, p->dt_bias, p->gate_lower_bound, p->beta_sigmoid,
                             p->beta_bf16)) != LA_OK)
        return st;
    ka.g = p->g;
    ka.g_st = p->g_stride_t;
    ka.g_sh = p->g_stride_h;
    ka.beta = p->beta;
    ka.b_st = p->beta_stride_t;
    ka.b_sh = p->beta_stride_h;
    ka.cu = p->cu_seqlens;
    ka.cu64 = p->cu_seqlens_bits == 64;
    ka.T = p->T;
    ka.N = p->N;
    ka.HK = p->HK;
    ka.HV = p->HV;
    ka.K = p->K;
    ka.V = p->V;
    ka.group = p->HV / p->HK;
    ka.scale = p->scale > 0.f ? p->scale : 1.0f / std::sqrt(static_cast<float>(p->K));
    ka.l2norm = p->use_qk_l2norm != 0;
    ka.s0 = p->d_final_state;
    ka.final_state = p->d_state;
    ka.tiles_per_head = 1;
    ka.num_units = static_cast<int64_t>(p->N) * p->HV;
    ka.hdr = pa.hdr;
    ka.order = pa.order;
    ka.ckpt_off = pa.ckpt_off;
    ka.chunk_off = pa.chunk_off;
    ka.chunk_seq = pa.chunk_seq;
    ka.wy = wb + GL.wy;
    ka.user_status = p->status;
    ka.wait_budget_ns = kWaitBudgetNs;
    ka.gdp_n = 1;
    if (const uint64_t b = g_test_wait_budget_ns.load(std::memory_order_relaxed)) ka.wait_budget_ns = b;
    if (ka.num_units == 0) return LA_OK;

    CUtensorMap qm, km, dom, wm;
    if ((st = make_map(&km, p->k, p->T, p->HK, p->K, p->k_stride_t, p->k_stride_h)) != LA_OK) return st;
    if ((st = make_map(&qm, p->q, p->T, p->HK, p->K, p->q_stride_t, p->q_stride_h)) != LA_OK) return st;
    if ((st = make_map(&dom, p->d_o, p->T, p->HV, p->V, p->d_o_stride_t, p->d_o_stride_h)) != LA_OK) return st;
    if ((st = make_map(&wm, ka.wy, 136, GL.items, 64, 64, static_cast<int64_t>(la::kWyRecordBytes / 2))) != LA_OK)
        return st;
    cudaEvent_t ev0 = t_timing_start, ev1 = t_timing_stop;
    t_timing_start = t_timing_stop = nullptr;
    if (ev0 && cudaEventRecord(ev0, s) != cudaSuccess) return LA_ERR_CUDA;
    ChunkArgs kw = ka;
    kw.num_units = GL.items;  // the bound on (chunk, head) items
    if (la::launch_wy_kernel(kw, qm, km, wm, la::kWyFwd, s) != cudaSuccess) return LA_ERR_CUDA;
    if (la::launch_grad(ka, qm, km, dom, wm, s) != cudaSuccess) return LA_ERR_CUDA;
    if (ev1 && cudaEventRecord(ev1, s) != cudaSuccess) return LA_ERR_CUDA;
    return LA_OK;
}
}  // namespace

la_status gdn_summary_bwd(const la_gdn_summary_bwd_params* p, void* stream) {
    if (!p) return LA_ERR_INVALID_ARG;
    Common c{p->T, p->N, p->HK, p->HV, p->K, p->V, p->cu_seqlens, p->cu_seqlens_bits, p->g, p->beta,
             p->beta_bf16 ? 2 : 4};
    la_status st = check_common(c);
    if (st != LA_OK) return st;
    la::BwdArgs b;
    std::memset(&b, 0, sizeof(b));
    if ((st = set_bwd_transforms(b, p->gate_mode, p->a_log, p->dt_bias, p->gate_lower_bound, p->beta_sigmoid,
                                 p->beta_bf16)) != LA_OK)
        return st;
    if (!p->d_state || !aligned(p->d_state, 4)) return LA_ERR_INVALID_ARG;
    if (p->d_final_state && !aligned(p->d_final_state, 4)) return LA_ERR_INVALID_ARG;
    if (p->T > 0) {
        if ((st = check_tma_operand(p->q, p->q_stride_t, p->q_stride_h, p->HK)) != LA_OK) return st;
        if ((st = check_tma_operand(p->k, p->k_stride_t, p->k_stride_h, p->HK)) != LA_OK) return st;
        if (!p->d_o || !aligned(p->d_o, 2)) return LA_ERR_INVALID_ARG;
    }
    // On the tensor cores when the workspace has room for the forward's WY records: the WY pass,
    // then the state-gradient pass (gdn_grad.cu); otherwise the tile kernel's state-only mode.
    {
        const int32_t passes = g_test_fwd_passes.load(std::memory_order_relaxed);
        const la::SplitLayout GL = la::split_layout(p->T, p->N, p->HV);
        bool two = passes != 1 && p->T > 0 && GL.items < (int64_t(1) << 31) && aligned(p->d_o, 16) &&
                   p->d_o_stride_t % 8 == 0 && (p->HV == 1 || p->d_o_stride_h % 8 == 0);
        void* w2 = nullptr;
        if (two) {
            if (p->workspace) {
                two = p->workspace_bytes >= GL.total && aligned(p->workspace, 256);
                w2 = p->workspace;
            } else {
                two = internal_workspace(GL.total, static_cast<cudaStream_t>(stream), &w2) == LA_OK;
            }
        }
        if (two) return summary_bwd_two_pass(p, GL, static_cast<uint8_t*>(w2), static_cast<cudaStream_t>(stream));
    }
    const SumBwdLayout SL = sum_bwd_layout(p->N, p->HV, p->K, p->V);
    void* ws = p->workspace;
    if (ws) {
        if (p->workspace_bytes < SL.total || !aligned(ws, 256)) return LA_ERR_WORKSPACE;
    } else if ((st = internal_workspace(SL.total, static_cast<cudaStream_t>(stream), &ws)) != LA_OK) {
        return st;
    }
    uint8_t* wb = static_cast<uint8_t*>(ws);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const la::WorkspaceLayout PL = la::ws_layout(p->N);
    // the prologue validates cu_seqlens into the status word the kernel reads first
    PrologueArgs pa;
    pa.cu = p->cu_seqlens;
    pa.chunk_off = nullptr;
    pa.chunk_rows = 1;
    pa.cu64 = p->cu_seqlens_bits == 64;
    pa.T = p->T;
    pa.N = p->N;
    pa.ckpt_n = la::kChunk;
    pa.hdr = reinterpret_cast<la::WsHeader*>(wb + SL.pro);
    pa.order = reinterpret_cast<int32_t*>(wb + SL.pro + PL.order);
    pa.ckpt_off = reinterpret_cast<int64_t*>(wb + SL.pro + PL.ckpt_off);
    pa.keys = reinterpret_cast<uint64_t*>(wb + SL.pro + PL.keys);
    pa.user_status = p->status;
    if (la::launch_prologue(pa, s) != cudaSuccess) return LA_ERR_CUDA;
    b.q = static_cast<const uint16_t*>(p->q); b.q_st = p->q_stride_t; b.q_sh = p->q_stride_h;
    b.k = static_cast<const uint16_t*>(p->k); b.k_st = p->k_stride_t; b.k_sh = p->k_stride_h;
    b.g = p->g; b.g_st = p->g_stride_t; b.g_sh = p->g_stride_h;
    b.beta = p->beta; b.b_st = p->beta_stride_t; b.b_sh = p->beta_stride_h;
    b.cu = p->cu_seqlens; b.cu64 = p->cu_seqlens_bits == 64;
    b.T = p->T; b.N = p->N; b.HK = p->HK; b.HV = p->HV; b.K = p->K; b.V = p->V; b.group = p->HV / p->HK;
    b.scale = p->scale > 0.f ? p->scale : 1.0f / std::sqrt(static_cast<float>(p->K));
    b.l2norm = p->use_qk_l2norm != 0;
    b.dout = static_cast<const uint16_t*>(p->d_o); b.do_st = p->d_o_stride_t; b.do_sh = p->d_o_stride_h;
    b.dfinal = p->d_final_state;
    b.ckpt_off = reinterpret_cast<const int64_t*>(wb + SL.pro + PL.ckpt_off);
    b.hdr = reinterpret_cast<const la::WsHeader*>(wb + SL.pro);
    b.dS_work = reinterpret_cast<float*>(wb + SL.ds);
    b.ds0 = p->d_state;
    b.vo_async = aligned(p->d_o, 4) && p->d_o_stride_t % 2 == 0 && (p->HV == 1 || p->d_o_stride_h % 2 == 0);
    b.state_only = 1;
    cudaEvent_t ev0 = t_timing_start, ev1 = t_timing_stop;
    t_timing_start = t_timing_stop = nullptr;
    if (ev0 && cudaEventRecord(ev0, s) != cudaSuccess) return LA_ERR_CUDA;
    if (la::launch_bwd(b, s) != cudaSuccess) return LA_ERR_CUDA;
    if (ev1 && cudaEventRecord(ev1, s) != cudaSuccess) return LA_ERR_CUDA;
    return LA_OK;
}

la_status gdn_compose_spans(const la_gdn_compose_params* p, void* stream) {
    if (!p || !p->out || p->R < 0 || p->HO < 1) return LA_ERR_INVALID_ARG;
    if ((p->K != 64 && p->K != 128) || (p->V != 64 && p->V != 128)) return LA_ERR_UNSUPPORTED;
    if (p->R > 0 && (!p->transitions || !p->terms)) return LA_ERR_INVALID_ARG;
    if (!aligned(p->out, 4) || !aligned(p->transitions, 4) || !aligned(p->terms, 4) || !aligned(p->start, 4))
        return LA_ERR_INVALID_ARG;
    la::ComposeArgs a;
    a.R = p->R;
    a.HO = p->HO;
    a.K = p->K;
    a.V = p->V;
    a.transitions = p->transitions;
    a.terms = p->terms;
    a.start = p->start;
    a.out = p->out;
    a.backward = p->backward != 0;
    return la::launch_compose(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

la_status gdn_summary(const la_gdn_summary_params* p, void* stream) {
    if (!p) return LA_ERR_INVALID_ARG;
    Common c{p->T, p->N, p->HK, p->HV, p->K, p->V, p->cu_seqlens, p->cu_seqlens_bits, p->g, p->beta,
             p->beta_bf16 ? 2 : 4};
    la_status st = check_common(c);
    if (st != LA_OK) return st;
    if (p->T > 0) {
        if ((st = check_tma_operand(p->k, p->k_stride_t, p->k_stride_h, p->HK)) != LA_OK) return st;
        if ((st = check_tma_operand(p->v, p->v_stride_t, p->v_stride_h, p->HV)) != LA_OK) return st;
    }
    if (!p->end_state || !p->transition) return LA_ERR_INVALID_ARG;
    if (!aligned(p->end_state, 4) || !aligned(p->transition, 16)) return LA_ERR_INVALID_ARG;
    if (p->start_state) {
        if (p->start_state_dtype != LA_DTYPE_F32 && p->start_state_dtype != LA_DTYPE_BF16) return LA_ERR_UNSUPPORTED;
        if (!aligned(p->start_state, p->start_state_dtype == LA_DTYPE_F32 ? 4 : 2)) return LA_ERR_INVALID_ARG;
    }
    ChunkArgs ka;
    std::memset(&ka, 0, sizeof(ka));
    ka.g_st = p->g_stride_t;
    ka.g_sh = p->g_stride_h;
    ka.b_st = p->beta_stride_t;
    ka.b_sh = p->beta_stride_h;
    ka.scale = 1.f;
    ka.l2norm = p->use_qk_l2norm != 0;
    ka.s0 = p->start_state;
    ka.s0_bf16 = p->start_state_dtype == LA_DTYPE_BF16;
    ka.final_state = p->end_state;
    ka.transition = p->transition;
    ka.tiles_per_head = 2;
    if ((st = set_transforms(ka, p->gate_mode, p->a_log, p->dt_bias, p->gate_lower_bound, p->beta_sigmoid,
                             p->beta_bf16)) != LA_OK)
        return st;
    return run(c, ka, nullptr, 0, 0, p->k, p->k_stride_t, p->k_stride_h, p->v, p->v_stride_t, p->v_stride_h, 0,
               p->workspace, p->workspace_bytes, p->status, la::kModeSummary, static_cast<cudaStream_t>(stream));
}

la_status gdn_fwd_static_workspace(const la_gdn_fwd_params* p, void* stream) {
    if (!p) return LA_ERR_INVALID_ARG;
    if (p->workspace) return LA_ERR_INVALID_ARG;  // the scratch is the library's own array
    if (p->N < 0) return LA_ERR_INVALID_ARG;
    // GDP beyond 64 updates per token materialises its timeline in a scratch that grows with T
    if (p->num_householder > la::kChunk) return LA_ERR_UNSUPPORTED;
    if (p->N > kStaticMaxSeqs || la::ws_layout(p->N).total > kStaticScratchBytes) return LA_ERR_WORKSPACE;
    void* scratch = nullptr;
    la_status st = static_scratch_address(&scratch);
    if (st != LA_OK) return st;
    la_gdn_fwd_params q = *p;
    q.workspace = scratch;
    q.workspace_bytes = kStaticScratchBytes;
    return gdn_fwd(&q, stream);
}

size_t la_gdn_workspace_bytes(int32_t N, int32_t summary) {
    (void)summary;
    return la::ws_layout(N).total;
}

size_t la_gdn_fwd_split_workspace_bytes(int64_t T, int32_t N, int32_t HV) {
    if (T < 0 || N < 0 || HV <= 0) return 0;
    return la::split_layout(T, N, HV).total;
}

la_status la_checkpoint_rows(const void* cu_seqlens_host, int32_t idx_bits, int32_t N, int64_t n, int64_t* rows_out) {
    if (!cu_seqlens_host || !rows_out || n <= 0 || N < 0 || (idx_bits != 32 && idx_bits != 64))
        return LA_ERR_INVALID_ARG;
    int64_t rows = 0;
    for (int32_t i = 0; i < N; ++i) {
        int64_t a, b;
        if (idx_bits == 64) {
            a = static_cast<const int64_t*>(cu_seqlens_host)[i];
            b = static_cast<const int64_t*>(cu_seqlens_host)[i + 1];
        } else {
            a = static_cast<const int32_t*>(cu_seqlens_host)[i];
            b = static_cast<const int32_t*>(cu_seqlens_host)[i + 1];
        }
        if (b < a) return LA_ERR_INVALID_ARG;
        rows += (b - a + n - 1) / n;
    }
    *rows_out = rows;
    return LA_OK;
}

la_status la_read_status(const int32_t* device_status, void* stream, int32_t* out) {
    if (!device_status || !out) return LA_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return LA_ERR_CUDA;
    if (cudaMemcpy(out, device_status, sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess) return LA_ERR_CUDA;
    return LA_OK;
}

la_status la_test_set_wait_hooks(int32_t skip_tile_load, uint64_t wait_budget_ns) {
    g_test_skip_tile_load.store(skip_tile_load != 0 ? 1 : 0, std::memory_order_relaxed);
    g_test_wait_budget_ns.store(wait_budget_ns, std::memory_order_relaxed);
    return LA_OK;
}

la_status la_test_set_fwd_passes(int32_t passes) {
    if (passes < 0 || passes > 2) return LA_ERR_INVALID_ARG;
    g_test_fwd_passes.store(passes, std::memory_order_relaxed);
    return LA_OK;
}

la_status la_test_set_fwd_pieces(int32_t pieces) {
    if (pieces < 0 || pieces > 16) return LA_ERR_INVALID_ARG;
    g_test_fwd_pieces.store(pieces, std::memory_order_relaxed);
    return LA_OK;
}

la_status la_set_kernel_timing_events(void* start_event, void* stop_event) {
    t_timing_start = static_cast<cudaEvent_t>(start_event);
    t_timing_stop = static_cast<cudaEvent_t>(stop_event);
    return LA_OK;
}

const char* la_status_string(la_status s) {
    switch (s) {
        case LA_OK: return "ok";
        case LA_ERR_INVALID_ARG: return "invalid argument (pointer, shape, stride or alignment)";
        case LA_ERR_UNSUPPORTED: return "unsupported configuration (head dims, head grouping or dtype)";
        case LA_ERR_CUDA: return "a CUDA call failed";
        case LA_ERR_BAD_SEQLENS: return "cu_seqlens must start at 0, be nondecreasing and end at T";
        case LA_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out";
        case LA_ERR_WORKSPACE: return "workspace too small or not 256-byte aligned";
        case LA_ERR_BAD_STATE_INDEX: return "a state_indices entry lies outside the state pool";
    }
    return "unknown status";
}

int32_t la_version(void) { return 100; }

}  // extern "C"
