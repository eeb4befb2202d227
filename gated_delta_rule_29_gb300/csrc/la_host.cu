// la_host.cu -- gdn_fwd on host buffers (the C ABI entry gdn_fwd_host).
//
// The packed batch is cut into token ranges: runs of whole sequences, and sequences longer
// than a range cut into pieces at multiples of the range length P.  P is a multiple of the
// 64-token chunk and of the checkpoint cadence, so a piece continues the chunk sequence of the
// one before it from the exact fp32 state that one ended in, and the result is bitwise that
// of one gdn_fwd call (a sequence's results do not depend on the batch around it).  For each
// range, in packed order: its inputs are copied in on the copy-in stream, its forward runs on
// one of eight compute streams once they have arrived (the pieces of one sequence share a
// stream, so they run in order), and its outputs are copied out on the copy-out stream once
// the forward is done.  The streams, a pinned metadata buffer and its event are owned per
// device.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/liblinattn.h"

namespace {

constexpr int kHostStreams = 8;
constexpr int64_t kChunk = 64;

struct Range {
    int64_t t_a, t_b;
    int32_t a, b, piece, last;
};

int64_t cu_at(const void* cu, int32_t bits, int64_t i) {
    return bits == 64 ? static_cast<const int64_t*>(cu)[i] : static_cast<const int32_t*>(cu)[i];
}

int64_t gcd64(int64_t a, int64_t b) {
    while (b) {
        const int64_t t = a % b;
        a = b;
        b = t;
    }
    return a;
}

// The ranges for a validated cu_seqlens; returns P.
int64_t make_plan(const void* cu, int32_t bits, int32_t N, int32_t ranges, int64_t n, std::vector<Range>& out) {
    const int64_t total = N > 0 ? cu_at(cu, bits, N) : 0;
    const int64_t unit = n > 0 ? kChunk / gcd64(kChunk, n) * n : kChunk;
    const int64_t parts = ranges > 0 ? ranges : 1;
    const int64_t target = total > 0 ? (total + parts - 1) / parts : 1;
    const int64_t P = std::max(unit, (target + unit - 1) / unit * unit);
    int64_t t = 0, run_t = 0;
    int32_t run_a = 0;
    for (int32_t i = 0; i < N; ++i) {
        const int64_t L = cu_at(cu, bits, i + 1) - cu_at(cu, bits, i);
        if (L > P) {
            if (i > run_a) out.push_back({run_t, t, run_a, i, -1, 1});
            const int64_t np = (L + P - 1) / P;
            for (int64_t pc = 0; pc < np; ++pc)
                out.push_back({t + pc * P, t + std::min(L, (pc + 1) * P), i, i + 1, static_cast<int32_t>(pc),
                               pc == np - 1 ? 1 : 0});
            t += L;
            run_a = i + 1;
            run_t = t;
            continue;
        }
        if (t + L - run_t > P && i > run_a) {
            out.push_back({run_t, t, run_a, i, -1, 1});
            run_a = i;
            run_t = t;
        }
        t += L;
    }
    if (N > run_a) out.push_back({run_t, t, run_a, N, -1, 1});
    return P;
}

bool seqlens_ok(const void* cu, int32_t bits, int32_t N, int64_t T) {
    if (cu_at(cu, bits, 0) != 0 || cu_at(cu, bits, N) != T) return false;
    for (int32_t i = 0; i < N; ++i)
        if (cu_at(cu, bits, i + 1) < cu_at(cu, bits, i)) return false;
    return true;
}

size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// Everything the call derives from its parameters: the plan, the checkpoint rows and the
// staging layout (byte offsets into the caller's device buffer).
struct HostPlan {
    std::vector<Range> parts;
    std::vector<int64_t> row_off;  // [N + 1] checkpoint row of each sequence's first entry
    std::vector<int32_t> slot;     // [N] hand-over slot of a cut sequence, else -1
    int32_t nlong = 0;
    size_t cu_count = 0;           // int32 entries of all ranges' cu_seqlens
    size_t q, k, v, g, beta, s0, o, fin, ck, mid, meta, ws, ws_each, total;
    size_t meta_bytes;             // pinned metadata: cu arrays, a_log, dt_bias
};

la_status make_host_plan(const la_gdn_fwd_host_params* hp, HostPlan& P) {
    if (!hp) return LA_ERR_INVALID_ARG;
    const la_gdn_fwd_params& f = hp->fwd;
    if (f.N < 0 || f.T < 0 || f.HK <= 0 || f.HV <= 0 || hp->ranges < 1) return LA_ERR_INVALID_ARG;
    if ((f.K != 64 && f.K != 128) || (f.V != 64 && f.V != 128)) return LA_ERR_UNSUPPORTED;
    if (f.HV % f.HK != 0 || f.T >= (int64_t(1) << 31) - 64) return LA_ERR_UNSUPPORTED;
    if (f.num_householder > 1 || f.state_indices) return LA_ERR_UNSUPPORTED;
    if (f.cu_seqlens_bits != 32 && f.cu_seqlens_bits != 64) return LA_ERR_INVALID_ARG;
    if (!f.cu_seqlens) return LA_ERR_INVALID_ARG;
    if (!seqlens_ok(f.cu_seqlens, f.cu_seqlens_bits, f.N, f.T)) return LA_ERR_BAD_SEQLENS;
    if (f.checkpoints && (f.checkpoint_every_n <= 0 || f.checkpoint_every_n % kChunk != 0)) return LA_ERR_INVALID_ARG;
    const int64_t n = f.checkpoints ? f.checkpoint_every_n : 0;
    make_plan(f.cu_seqlens, f.cu_seqlens_bits, f.N, hp->ranges, n, P.parts);
    P.row_off.assign(static_cast<size_t>(f.N) + 1, 0);
    for (int32_t i = 0; i < f.N; ++i) {
        const int64_t L = cu_at(f.cu_seqlens, f.cu_seqlens_bits, i + 1) - cu_at(f.cu_seqlens, f.cu_seqlens_bits, i);
        P.row_off[i + 1] = P.row_off[i] + (n ? (L + n - 1) / n : 0);
    }
    P.slot.assign(static_cast<size_t>(f.N), -1);
    P.cu_count = 0;
    for (const Range& r : P.parts) {
        if (r.piece == 0) P.slot[r.a] = P.nlong++;
        P.cu_count += r.piece < 0 ? static_cast<size_t>(r.b - r.a + 1) : 2;
    }
    const size_t T = static_cast<size_t>(f.T), N = static_cast<size_t>(f.N);
    const size_t HK = f.HK, HV = f.HV, K = f.K, V = f.V;
    const size_t state = HV * K * V;
    const size_t s0_es = f.initial_state_dtype == LA_DTYPE_BF16 ? 2 : 4;
    const size_t ck_es = f.checkpoint_dtype == LA_DTYPE_BF16 ? 2 : 4;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += up256(bytes);
        return at;
    };
    P.q = take(T * HK * K * 2);
    P.k = take(T * HK * K * 2);
    P.v = take(T * HV * V * 2);
    P.g = take(T * HV * 4);
    P.beta = take(T * HV * (f.beta_bf16 ? 2 : 4));
    P.s0 = take(f.initial_state ? N * state * s0_es : 0);
    P.o = take(T * HV * V * 2);
    P.fin = take(f.final_state ? N * state * 4 : 0);
    P.ck = take(f.checkpoints ? static_cast<size_t>(P.row_off[f.N]) * state * ck_es : 0);
    P.mid = take(static_cast<size_t>(P.nlong) * 2 * state * 4);
    P.meta_bytes = P.cu_count * 4 + (f.gate_mode == LA_GATE_SOFTPLUS ? 2 * HV * 4 : 0);
    P.meta = take(P.meta_bytes);
    // each compute stream's workspace has room for the two-pass forward of the largest range
    P.ws_each = up256(la_gdn_workspace_bytes(f.N, 0));
    for (const Range& r : P.parts) {
        const int32_t nr = r.piece < 0 ? r.b - r.a : 1;
        const size_t need = la_gdn_fwd_split_workspace_bytes(r.t_b - r.t_a, nr, f.HV);
        if (up256(need) > P.ws_each) P.ws_each = up256(need);
    }
    P.ws = take(P.ws_each * kHostStreams);
    P.total = off;
    return LA_OK;
}

struct HostPipe {
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr, cs[kHostStreams] = {};
    void* meta = nullptr;  // pinned
    size_t meta_cap = 0;
    cudaEvent_t meta_ev = nullptr;
    bool meta_pending = false;
    // the end of the last call that used each staging buffer
    std::vector<std::pair<const void*, cudaEvent_t>> done;
};
std::mutex g_host_mutex;
HostPipe g_host[128];

la_status pipe_for_device(HostPipe** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return LA_ERR_CUDA;
    HostPipe& hp = g_host[dev];
    if (!hp.ready) {
        if (cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking) != cudaSuccess) return LA_ERR_CUDA;
        if (cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking) != cudaSuccess) return LA_ERR_CUDA;
        for (int x = 0; x < kHostStreams; ++x)
            if (cudaStreamCreateWithFlags(&hp.cs[x], cudaStreamNonBlocking) != cudaSuccess) return LA_ERR_CUDA;
        if (cudaEventCreateWithFlags(&hp.meta_ev, cudaEventDisableTiming) != cudaSuccess) return LA_ERR_CUDA;
        hp.ready = true;
    }
    *out = &hp;
    return LA_OK;
}

// One event recorded on `from` that `to` waits for (destroyed at once: its resources go when
// it completes).
la_status chain(cudaStream_t from, cudaStream_t to) {
    cudaEvent_t e;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return LA_ERR_CUDA;
    const bool ok = cudaEventRecord(e, from) == cudaSuccess && cudaStreamWaitEvent(to, e, 0) == cudaSuccess;
    cudaEventDestroy(e);
    return ok ? LA_OK : LA_ERR_CUDA;
}

la_status copy(void* dst, const void* src, size_t bytes, cudaMemcpyKind kind, cudaStream_t s) {
    if (bytes == 0) return LA_OK;
    return cudaMemcpyAsync(dst, src, bytes, kind, s) == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

bool contiguous3(int64_t st, int64_t sh, int32_t H, int32_t D) { return st == int64_t(H) * D && (H == 1 || sh == D); }
bool contiguous2(int64_t st, int64_t sh, int32_t H) { return st == H && (H == 1 || sh == 1); }

}  // namespace

extern "C" {

int32_t la_gdn_fwd_host_plan(const void* cu_seqlens_host, int32_t idx_bits, int32_t N, int32_t ranges,
                             int64_t checkpoint_every_n, int64_t* out, int32_t max_ranges, int64_t* piece_tokens) {
    if (!cu_seqlens_host || N < 0 || ranges < 1 || checkpoint_every_n < 0 || max_ranges < 0 ||
        (idx_bits != 32 && idx_bits != 64) || (max_ranges > 0 && !out))
        return -1;
    if (!seqlens_ok(cu_seqlens_host, idx_bits, N, cu_at(cu_seqlens_host, idx_bits, N))) return -1;
    std::vector<Range> parts;
    const int64_t P = make_plan(cu_seqlens_host, idx_bits, N, ranges, checkpoint_every_n, parts);
    if (piece_tokens) *piece_tokens = P;
    for (size_t i = 0; i < parts.size() && i < static_cast<size_t>(max_ranges); ++i) {
        const Range& r = parts[i];
        const int64_t row[6] = {r.t_a, r.t_b, r.a, r.b, r.piece, r.last};
        std::memcpy(out + 6 * i, row, sizeof(row));
    }
    return static_cast<int32_t>(parts.size());
}

size_t la_gdn_fwd_host_staging_bytes(const la_gdn_fwd_host_params* p) {
    HostPlan P;
    return make_host_plan(p, P) == LA_OK ? P.total : 0;
}

la_status gdn_fwd_host(const la_gdn_fwd_host_params* hp, void* stream) {
    HostPlan P;
    la_status st = make_host_plan(hp, P);
    if (st != LA_OK) return st;
    const la_gdn_fwd_params& f = hp->fwd;
    if (f.T > 0) {
        if (!f.q || !f.k || !f.v || !f.g || !f.beta || !f.o) return LA_ERR_INVALID_ARG;
        if (!contiguous3(f.q_stride_t, f.q_stride_h, f.HK, f.K) || !contiguous3(f.k_stride_t, f.k_stride_h, f.HK, f.K) ||
            !contiguous3(f.v_stride_t, f.v_stride_h, f.HV, f.V) || !contiguous3(f.o_stride_t, f.o_stride_h, f.HV, f.V) ||
            !contiguous2(f.g_stride_t, f.g_stride_h, f.HV) || !contiguous2(f.beta_stride_t, f.beta_stride_h, f.HV))
            return LA_ERR_INVALID_ARG;
    }
    if (f.gate_mode == LA_GATE_SOFTPLUS && (!f.a_log || !f.dt_bias)) return LA_ERR_INVALID_ARG;
    if (!hp->staging || hp->staging_bytes < P.total || (reinterpret_cast<uintptr_t>(hp->staging) & 255) != 0)
        return LA_ERR_WORKSPACE;
    std::lock_guard<std::mutex> lock(g_host_mutex);
    HostPipe* pipe = nullptr;
    if ((st = pipe_for_device(&pipe)) != LA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* dev = static_cast<uint8_t*>(hp->staging);
    const int64_t HK = f.HK, HV = f.HV, K = f.K, V = f.V;
    const size_t state = static_cast<size_t>(HV * K * V);
    const size_t s0_es = f.initial_state_dtype == LA_DTYPE_BF16 ? 2 : 4;
    const size_t ck_es = f.checkpoint_dtype == LA_DTYPE_BF16 ? 2 : 4;
    const size_t b_es = f.beta_bf16 ? 2 : 4;

    // metadata (every range's cu_seqlens, the softplus gate's parameters) through the pinned
    // buffer: wait for the previous call's copy of it, refill, one copy
    if (pipe->meta_pending) {
        if (cudaEventSynchronize(pipe->meta_ev) != cudaSuccess) return LA_ERR_CUDA;
        pipe->meta_pending = false;
    }
    if (pipe->meta_cap < P.meta_bytes) {
        if (pipe->meta) cudaFreeHost(pipe->meta);
        pipe->meta = nullptr;
        pipe->meta_cap = 0;
        const size_t cap = std::max<size_t>(P.meta_bytes, 1 << 16);
        if (cudaHostAlloc(&pipe->meta, cap, cudaHostAllocDefault) != cudaSuccess) return LA_ERR_CUDA;
        pipe->meta_cap = cap;
    }
    std::vector<size_t> cu_at_part(P.parts.size());
    {
        int32_t* m = static_cast<int32_t*>(pipe->meta);
        size_t x = 0;
        for (size_t pi = 0; pi < P.parts.size(); ++pi) {
            const Range& r = P.parts[pi];
            cu_at_part[pi] = x;
            if (r.piece < 0) {
                const int64_t base = cu_at(f.cu_seqlens, f.cu_seqlens_bits, r.a);
                for (int32_t i = r.a; i <= r.b; ++i)
                    m[x++] = static_cast<int32_t>(cu_at(f.cu_seqlens, f.cu_seqlens_bits, i) - base);
            } else {
                m[x++] = 0;
                m[x++] = static_cast<int32_t>(r.t_b - r.t_a);
            }
        }
        if (f.gate_mode == LA_GATE_SOFTPLUS) {
            std::memcpy(m + P.cu_count, f.a_log, HV * sizeof(float));
            std::memcpy(m + P.cu_count + HV, f.dt_bias, HV * sizeof(float));
        }
    }
    // The copies in wait for the end of the last call that used this staging buffer (its device
    // copies, scratch and hand-over slots are about to be overwritten); a staging buffer not seen
    // before orders the call after the caller's stream.  Everything else follows from the copies
    // in by events, and the internal streams are FIFO across calls.
    cudaEvent_t* done_ev = nullptr;
    for (auto& e : pipe->done)
        if (e.first == hp->staging) done_ev = &e.second;
    if (done_ev) {
        if (cudaStreamWaitEvent(pipe->h2d, *done_ev, 0) != cudaSuccess) return LA_ERR_CUDA;
    } else {
        if (pipe->done.size() >= 64) {  // forget the oldest (a call on it is ordered by its caller's stream)
            cudaEventDestroy(pipe->done.front().second);
            pipe->done.erase(pipe->done.begin());
        }
        cudaEvent_t e;
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return LA_ERR_CUDA;
        pipe->done.emplace_back(hp->staging, e);
        done_ev = &pipe->done.back().second;
        if ((st = chain(s, pipe->h2d)) != LA_OK) return st;
    }
    if ((st = copy(dev + P.meta, pipe->meta, P.meta_bytes, cudaMemcpyHostToDevice, pipe->h2d)) != LA_OK) return st;
    if (cudaEventRecord(pipe->meta_ev, pipe->h2d) != cudaSuccess) return LA_ERR_CUDA;
    pipe->meta_pending = true;
    const int32_t* cu_d = reinterpret_cast<const int32_t*>(dev + P.meta);
    const float* alog_d = f.gate_mode == LA_GATE_SOFTPLUS ? reinterpret_cast<const float*>(dev + P.meta) + P.cu_count : nullptr;

    std::vector<int32_t> seq_stream(static_cast<size_t>(f.N), -1);
    int32_t next_stream = 0;
    const uint8_t* hq = static_cast<const uint8_t*>(f.q);
    const uint8_t* hk = static_cast<const uint8_t*>(f.k);
    const uint8_t* hv = static_cast<const uint8_t*>(f.v);
    const uint8_t* hg = reinterpret_cast<const uint8_t*>(f.g);
    const uint8_t* hb = reinterpret_cast<const uint8_t*>(f.beta);
    const uint8_t* hs0 = static_cast<const uint8_t*>(f.initial_state);
    uint8_t* ho = static_cast<uint8_t*>(f.o);
    uint8_t* hfin = reinterpret_cast<uint8_t*>(f.final_state);
    uint8_t* hck = static_cast<uint8_t*>(f.checkpoints);
    const size_t qrow = HK * K * 2, vrow = HV * V * 2, grow = HV * 4, brow = HV * b_es;
    for (size_t pi = 0; pi < P.parts.size(); ++pi) {
        const Range& r = P.parts[pi];
        const size_t ta = static_cast<size_t>(r.t_a), nt = static_cast<size_t>(r.t_b - r.t_a);
        const size_t sa = static_cast<size_t>(r.a), ns = static_cast<size_t>(r.b - r.a);
        // copy in
        cudaStream_t in = pipe->h2d;
        if ((st = copy(dev + P.q + ta * qrow, hq + ta * qrow, nt * qrow, cudaMemcpyHostToDevice, in)) != LA_OK ||
            (st = copy(dev + P.k + ta * qrow, hk + ta * qrow, nt * qrow, cudaMemcpyHostToDevice, in)) != LA_OK ||
            (st = copy(dev + P.v + ta * vrow, hv + ta * vrow, nt * vrow, cudaMemcpyHostToDevice, in)) != LA_OK ||
            (st = copy(dev + P.g + ta * grow, hg + ta * grow, nt * grow, cudaMemcpyHostToDevice, in)) != LA_OK ||
            (st = copy(dev + P.beta + ta * brow, hb + ta * brow, nt * brow, cudaMemcpyHostToDevice, in)) != LA_OK)
            return st;
        if (hs0 && r.piece <= 0 &&
            (st = copy(dev + P.s0 + sa * state * s0_es, hs0 + sa * state * s0_es, ns * state * s0_es,
                       cudaMemcpyHostToDevice, in)) != LA_OK)
            return st;
        // the forward of the range
        int32_t csi;
        if (r.piece >= 0) {
            if (seq_stream[r.a] < 0) seq_stream[r.a] = next_stream++ % kHostStreams;
            csi = seq_stream[r.a];
        } else {
            csi = static_cast<int32_t>(pi % kHostStreams);
        }
        cudaStream_t cs = pipe->cs[csi];
        if ((st = chain(in, cs)) != LA_OK) return st;
        la_gdn_fwd_params d = f;
        d.q = dev + P.q + ta * qrow;
        d.k = dev + P.k + ta * qrow;
        d.v = dev + P.v + ta * vrow;
        d.g = reinterpret_cast<const float*>(dev + P.g + ta * grow);
        d.beta = reinterpret_cast<const float*>(dev + P.beta + ta * brow);
        d.cu_seqlens = cu_d + cu_at_part[pi];
        d.cu_seqlens_bits = 32;
        d.T = static_cast<int64_t>(nt);
        d.N = static_cast<int32_t>(ns);
        d.o = dev + P.o + ta * vrow;
        d.a_log = alog_d;
        d.dt_bias = alog_d ? alog_d + HV : nullptr;
        d.workspace = dev + P.ws + static_cast<size_t>(csi) * P.ws_each;
        d.workspace_bytes = P.ws_each;
        uint8_t* mid = r.piece >= 0 ? dev + P.mid + static_cast<size_t>(P.slot[r.a]) * 2 * state * 4 : nullptr;
        if (r.piece <= 0) {
            d.initial_state = hs0 ? dev + P.s0 + sa * state * s0_es : nullptr;
        } else {
            d.initial_state = mid + static_cast<size_t>((r.piece - 1) % 2) * state * 4;
            d.initial_state_dtype = LA_DTYPE_F32;
        }
        if (r.piece < 0 || r.last) d.final_state = hfin ? reinterpret_cast<float*>(dev + P.fin + sa * state * 4) : nullptr;
        else d.final_state = reinterpret_cast<float*>(mid + static_cast<size_t>(r.piece % 2) * state * 4);
        int64_t r_a = P.row_off[r.a], r_b = P.row_off[r.b];
        if (r.piece >= 0 && f.checkpoints) {
            const int64_t n = f.checkpoint_every_n;
            const int64_t off = cu_at(f.cu_seqlens, f.cu_seqlens_bits, r.a);
            r_a = P.row_off[r.a] + (r.t_a - off) / n;
            r_b = P.row_off[r.a] + (r.t_b - off + n - 1) / n;
        }
        d.checkpoints = hck ? dev + P.ck + static_cast<size_t>(r_a) * state * ck_es : nullptr;
        if ((st = gdn_fwd(&d, cs)) != LA_OK) return st;
        // copy out
        cudaStream_t out = pipe->d2h;
        if ((st = chain(cs, out)) != LA_OK) return st;
        if ((st = copy(ho + ta * vrow, dev + P.o + ta * vrow, nt * vrow, cudaMemcpyDeviceToHost, out)) != LA_OK) return st;
        if (hfin && (r.piece < 0 || r.last) &&
            (st = copy(hfin + sa * state * 4, dev + P.fin + sa * state * 4, ns * state * 4, cudaMemcpyDeviceToHost,
                       out)) != LA_OK)
            return st;
        if (hck && r_b > r_a &&
            (st = copy(hck + static_cast<size_t>(r_a) * state * ck_es, dev + P.ck + static_cast<size_t>(r_a) * state * ck_es,
                       static_cast<size_t>(r_b - r_a) * state * ck_es, cudaMemcpyDeviceToHost, out)) != LA_OK)
            return st;
    }
    // the caller's stream continues after the last copy out (which follows every forward)
    if (cudaEventRecord(*done_ev, pipe->d2h) != cudaSuccess) return LA_ERR_CUDA;
    return cudaStreamWaitEvent(s, *done_ev, 0) == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

}  // extern "C"
