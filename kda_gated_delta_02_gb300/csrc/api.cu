// api.cu -- the C ABI declared in include/kda.h: argument validation, the
// context-parallel plan, workspace carving and kernel launches.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "../../include/kda.h"
#include "kda_internal.h"

namespace {

constexpr int kChunk = 64;

inline bool aligned16(const void *p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool dim_ok(int d) { return d == 64 || d == 128; }

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// SM count of the current device (cached per device)
int sm_count() {
    static std::atomic<int> cached[64];
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return 152;  // GB300
    }
    n = cached[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 152;
    }
    cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

// value-tile width of the warp-level prefill kernel: the whole dv, except that
// a transition (whose augmented state has dk + dv columns) tiles by 64 when
// dk is 64
int prefill_dvt(int dk, int dv, bool transition) {
    int dvt = (dv % 128 == 0) ? 128 : 64;
    if (transition && (dk % dvt != 0)) dvt = 64;
    return dvt;
}

struct CpLayout {
    int seg_len = 0;
    int P_max = 0;
    size_t off_count = 0, off_table = 0, off_first = 0, off_M = 0, off_N = 0, off_Sin = 0, total = 0;
};

CpLayout cp_layout(int N, int T, int H, int dk, int dv, int cp_mode, int segment_len) {
    CpLayout L;
    if (cp_mode == KDA_CP_OFF || N <= 0 || H <= 0) return L;
    if (cp_mode == KDA_CP_AUTO) {
        const int sms = sm_count();
        const long units = (long)N * H;
        const long avg = T / (N > 0 ? N : 1);
        if (!(units * 2 <= sms && avg >= 16 * kChunk)) return L;
    }
    int seg = segment_len;
    if (seg <= 0) {
        const int sms = sm_count();
        // segments per sequence: at d = 128 the walks hold one block per SM,
        // so about one wave of (segment, head) units; else two per SM
        long target = (dk == 128 && dv == 128) ? (long)sms / ((long)N * H)
                                               : (2L * sms + (long)N * H - 1) / ((long)N * H);
        if (target < 1) target = 1;
        long per = (T / (N > 0 ? N : 1) + target - 1) / target;
        seg = (int)(((per + kChunk - 1) / kChunk) * kChunk);
        if (seg < 16 * kChunk) seg = 16 * kChunk;
    }
    L.seg_len = seg;
    L.P_max = T / seg + N;
    size_t o = 0;
    L.off_count = o;
    o = align256(o + 16);
    L.off_table = o;
    o = align256(o + (size_t)L.P_max * 16);
    L.off_first = o;
    o = align256(o + (size_t)(N + 1) * 4);
    L.off_M = o;
    o = align256(o + (size_t)L.P_max * H * dk * dk * 4);
    L.off_N = o;
    o = align256(o + (size_t)L.P_max * H * dk * dv * 4);
    L.off_Sin = o;
    o = align256(o + (size_t)L.P_max * H * dk * dv * 4);
    L.total = o;
    return L;
}

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA; }

// Opt-in launch timing: a pair of CUDA events on the launching stream around
// every kernel launch of the library while enabled (kda_kernel_timing_start /
// kda_kernel_timing_stop).
struct TimedLaunch {
    int kind;
    cudaEvent_t a, b;
};
std::atomic<bool> g_timing{false};
std::mutex g_timing_mu;
std::vector<TimedLaunch> g_timed;

template <class F>
cudaError_t timed_launch(int kind, cudaStream_t st, F &&launch) {
    if (!g_timing.load(std::memory_order_relaxed)) return launch();
    cudaEvent_t a = nullptr, b = nullptr;
    if (cudaEventCreate(&a) != cudaSuccess || cudaEventCreate(&b) != cudaSuccess) {
        if (a) cudaEventDestroy(a);
        cudaGetLastError();
        return launch();
    }
    cudaEventRecord(a, st);
    const cudaError_t e = launch();
    cudaEventRecord(b, st);
    std::lock_guard<std::mutex> lk(g_timing_mu);
    g_timed.push_back({kind, a, b});
    return e;
}

void drop_timed() {
    for (const TimedLaunch &t : g_timed) {
        cudaEventDestroy(t.a);
        cudaEventDestroy(t.b);
    }
    g_timed.clear();
}

// Two-kernel tcgen05 prefill (dk = dv = 128): workspace after the CP scratch =
// slot list | one item counter per piece | two carry states [2 tiles][H][128][128]
// f32 | operand blobs of one or two pieces of slots.
//
// With two blob buffers the pieces are pipelined: the chunk-local kernel of
// piece p + 1 runs while the walk of piece p holds its SMs, and fills every SM
// once the walk is done; piece p + 2 reuses piece p's buffer (run_split).
// Calls with few slots run as one piece, and so do calls whose walks alone
// have a CTA for every SM (units x heads >= SMs: nothing is left idle to
// overlap); a context-parallel call keeps all slots in one piece when the
// workspace allows (the transition pass's blobs then serve the replay).  kda_chunk_fwd_prep_workspace_size asks for the
// layout the call prefers, the blobs capped at 16 GiB; smaller workspaces get
// smaller pieces.
struct SplitLayout {
    int nslots = 0, piece = 0, nbuf = 1, pieces = 0;
    size_t off_list = 0, off_claim = 0, off_carry = 0, carry_stride = 0, off_blob = 0, buf_bytes = 0, total = 0;
};

constexpr size_t kSplitBlobCap = (size_t)16384 << 20;
constexpr int kPipePieces = 4;     // pieces of a pipelined call
constexpr int kPipeMinSlots = 64;  // fewer slots than this run as one piece

// whether a call of `units` units over H heads prefers pipelined pieces
bool pipe_wanted(int units, int T, int H, bool one_piece) {
    return !one_piece && T / kChunk + units >= kPipeMinSlots && (long)units * H < sm_count();
}

inline size_t blob_per_slot(int H) { return (size_t)H * kda::kChunkBlobBytes; }

// Layout with room for the blobs of `room` slots.  one_piece: all slots in one
// piece when they fit; nbuf_max: 1 for a caller that runs the pieces in order
// on one stream.
SplitLayout split_layout_slots(int units, int T, int H, long room, bool one_piece, int nbuf_max) {
    SplitLayout S;
    S.nslots = T / kChunk + units;
    const long n = S.nslots;
    const long want = pipe_wanted(units, T, H, one_piece) ? (n + kPipePieces - 1) / kPipePieces : n;
    long piece = 0;
    if (nbuf_max <= 1) {
        piece = room < n ? room : n;
    } else if (room >= n && want >= n) {
        piece = n;
    } else if (room >= 2) {
        piece = want < room / 2 ? want : room / 2;
        S.nbuf = 2;
    } else if (room >= 1) {
        piece = 1;
    }
    if (piece >= 1) {
        const long pieces = (n + piece - 1) / piece;
        S.piece = (int)((n + pieces - 1) / pieces);
        S.pieces = (int)pieces;
        if (S.pieces == 1) S.nbuf = 1;
    } else {
        S.nbuf = 0;
    }
    size_t o = 0;
    S.off_list = o;
    o = align256(o + (size_t)n * 8);
    S.off_claim = o;
    o = align256(o + (size_t)n * 4);
    S.off_carry = o;
    S.carry_stride = (size_t)2 * H * 128 * 128;  // floats per carry state
    o = align256(o + 2 * S.carry_stride * 4);
    S.off_blob = o;
    S.buf_bytes = (size_t)S.piece * blob_per_slot(H);
    o = align256(o + (size_t)S.nbuf * S.buf_bytes);
    S.total = o;
    return S;
}

// The layout kda_chunk_fwd_prep_workspace_size asks for.
SplitLayout split_layout_wanted(int units, int T, int H, bool one_piece) {
    const long n = T / kChunk + units;
    const long cap = (long)(kSplitBlobCap / blob_per_slot(H));
    const long want = pipe_wanted(units, T, H, one_piece) ? 2 * ((n + kPipePieces - 1) / kPipePieces) : n;
    return split_layout_slots(units, T, H, want < cap ? want : (cap < 1 ? 1 : cap), one_piece, 2);
}

// The layout that fits `bytes` of workspace (piece = 0: none fits).
SplitLayout split_layout_fit(int units, int T, int H, size_t bytes, bool one_piece) {
    const SplitLayout fixed = split_layout_slots(units, T, H, 0, one_piece, 2);  // list, counters, carries
    if (bytes < fixed.total) return fixed;
    return split_layout_slots(units, T, H, (long)((bytes - fixed.total) / blob_per_slot(H)), one_piece, 2);
}

// One pass of the two-kernel prefill over `units` units: the chunk list, then
// per piece the chunk-local kernel and the walk, all on `st`.  With two blob
// buffers the chunk-local kernel of piece p + 1 is a programmatic dependent
// launch of the walk of piece p: the walk lets it start as soon as all of the
// walk's CTAs are resident, so it runs on the SMs the walk leaves free and
// fills the rest when the walk ends.  It reads nothing the walk writes and
// writes the other buffer, whose last reader (the walk of piece p - 1)
// completed before the walk of piece p started; every walk is an ordinary
// launch, so it starts only after all earlier work on the stream.  With
// skip_prep the blobs of a single piece are already in place (written by an
// earlier pass with need_q set).
cudaError_t run_split(const kda::ChunkArgs &a, int units, unsigned char *ws, const SplitLayout &S, bool need_q,
                      bool skip_prep, cudaStream_t st) {
    int2 *list = reinterpret_cast<int2 *>(ws + S.off_list);
    int *claim = reinterpret_cast<int *>(ws + S.off_claim);
    float *carry = reinterpret_cast<float *>(ws + S.off_carry);
    unsigned char *blob = ws + S.off_blob;
    const int P = S.pieces;
    const bool overlap = S.nbuf == 2;
    cudaError_t e = cudaSuccess;
    if (!skip_prep) {
        e = cudaMemsetAsync(claim, 0, (size_t)P * sizeof(int), st);
        if (e == cudaSuccess)
            e = timed_launch(KDA_KERNEL_CHUNK_LIST, st, [&] { return kda::launch_chunk_list(a, units, S.nslots, list, st); });
    }
    for (int pc = 0; e == cudaSuccess && pc < P; ++pc) {
        const int s0 = pc * S.piece, s1 = s0 + S.piece < S.nslots ? s0 + S.piece : S.nslots;
        unsigned char *buf = blob + (size_t)(pc % (S.nbuf > 0 ? S.nbuf : 1)) * S.buf_bytes;
        if (!skip_prep)
            e = timed_launch(KDA_KERNEL_CHUNK_PREP, st, [&] {
                return kda::launch_chunk_prep(a, list, s0, s1, buf, need_q, claim + pc, overlap && pc > 0, st);
            });
        if (e == cudaSuccess)
            e = timed_launch(KDA_KERNEL_CHUNK_WALK, st, [&] {
                return kda::launch_chunk_walk(a, units, buf, s0, s1, carry + (size_t)(pc & 1) * S.carry_stride,
                                              carry + (size_t)((pc + 1) & 1) * S.carry_stride, st);
            });
    }
    return e;
}

// Chunk-kernel dispatch by shape: the tcgen05 / tensor-memory kernel for
// dk = dv = 128 with bf16 inputs, the warp-level kernel otherwise.
cudaError_t run_chunk(const kda::ChunkArgs &a, int units, bool bf, cudaStream_t st) {
    if (kda::chunk_tc_supported(a, bf))
        return timed_launch(KDA_KERNEL_CHUNK_TC, st, [&] { return kda::launch_chunk_tc(a, units, st); });
    return timed_launch(KDA_KERNEL_CHUNK_MMA, st, [&] {
        return kda::launch_chunk(a, units, prefill_dvt(a.dk, a.dv, a.mode == kda::MODE_TRANSITION), bf, st);
    });
}

}  // namespace

namespace {
// ---------------------------------------------------------------- host-buffer prefill
// Device workspace of kda_chunk_fwd_host: device copies of the inputs and
// outputs, then the two-kernel area for one piece of slots.
struct HostLayout {
    size_t off_q = 0, off_k = 0, off_v = 0, off_g = 0, off_b = 0, off_cu = 0, off_s0 = 0, off_o = 0, off_sf = 0;
    size_t off_area = 0, total = 0;
    bool pipelined = false;
    SplitLayout S;
};

HostLayout host_layout(int N, int T, int H, int dk, int dv, int in_dtype, int pieces) {
    HostLayout L;
    const size_t es = in_dtype == KDA_DTYPE_BF16 ? 2 : 4;
    size_t o = 0;
    L.off_q = o; o = align256(o + (size_t)T * H * dk * es);
    L.off_k = o; o = align256(o + (size_t)T * H * dk * es);
    L.off_v = o; o = align256(o + (size_t)T * H * dv * es);
    L.off_g = o; o = align256(o + (size_t)T * H * dk * 4);
    L.off_b = o; o = align256(o + (size_t)T * H * 4);
    L.off_cu = o; o = align256(o + (size_t)(N + 1) * 4);
    L.off_s0 = o; o = align256(o + (size_t)N * H * dk * dv * 4);
    L.off_o = o; o = align256(o + (size_t)T * H * dv * es);
    L.off_sf = o; o = align256(o + (size_t)N * H * dk * dv * 4);
    L.off_area = o;
    L.pipelined = in_dtype == KDA_DTYPE_BF16 && dk == 128 && dv == 128 && T > 0;
    if (L.pipelined) {
        const int nslots = T / kChunk + N;
        const int pc = pieces < 1 ? 1 : (pieces > nslots ? nslots : pieces);
        L.S = split_layout_slots(N, T, H, (nslots + pc - 1) / pc, false, 1);
        o += L.S.total;
    }
    L.total = align256(o);
    return L;
}

// Per-stream state of the host-buffer prefill: two copy streams per device.
struct CopyStreams {
    cudaStream_t in = nullptr, out = nullptr;
};
std::mutex g_copy_mu;
CopyStreams g_copy[64];

int copy_streams(CopyStreams *cs) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return KDA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_copy_mu);
    if (!g_copy[dev].in) {  // both streams or neither
        CopyStreams made;
        if (cudaStreamCreateWithFlags(&made.in, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&made.out, cudaStreamNonBlocking) != cudaSuccess) {
            if (made.in) cudaStreamDestroy(made.in);
            cudaGetLastError();
            return KDA_ERR_CUDA;
        }
        g_copy[dev] = made;
    }
    *cs = g_copy[dev];
    return KDA_OK;
}
}  // namespace

extern "C" {

const char *kda_status_string(int status) {
    switch (status) {
        case KDA_OK: return "ok";
        case KDA_ERR_INVALID_ARG: return "invalid argument";
        case KDA_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case KDA_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
        case KDA_ERR_WORKSPACE: return "workspace missing or too small";
        case KDA_ERR_CUDA: return "CUDA launch error";
        case KDA_ERR_SCRATCH_LIMIT: return "request exceeds the fixed scratch of the no-allocation entry point";
        default: return "unknown status";
    }
}

int kda_version(void) { return 100; }

size_t kda_chunk_fwd_workspace_size(int N, int T, int H, int dk, int dv, int cp_mode, int segment_len) {
    return cp_layout(N, T, H, dk, dv, cp_mode, segment_len).total;
}

size_t kda_chunk_fwd_prep_workspace_size(int N, int T, int H, int dk, int dv, int cp_mode, int segment_len) {
    const CpLayout L = cp_layout(N, T, H, dk, dv, cp_mode, segment_len);
    if (dk != 128 || dv != 128 || N < 1 || T < 0 || H < 1) return L.total;
    const int units = L.seg_len ? L.P_max : N;
    return align256(L.total) + split_layout_wanted(units, T, H, L.seg_len != 0).total;
}

int kda_chunk_fwd_plan(int N, int T, int H, int dk, int dv, int cp_mode, int segment_len) {
    return cp_layout(N, T, H, dk, dv, cp_mode, segment_len).seg_len;
}

namespace {
int chunk_fwd_impl(const void *q, const void *k, const void *v, const float *g, const float *beta,
                   const int32_t *cu_seqlens, int N, int T, int H, int dk, int dv,
                   const float *initial_state, float *final_state, void *o, float scale, float g_min,
                   int in_dtype, int cp_mode, int segment_len, void *workspace, size_t workspace_bytes,
                   int ckpt_every, int ckpt_count, float *ckpt, uint32_t *status, void *stream) {
    if (N < 1 || T < 0 || H < 1) return KDA_ERR_INVALID_ARG;
    if (!dim_ok(dk) || !dim_ok(dv)) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (in_dtype != KDA_DTYPE_BF16 && in_dtype != KDA_DTYPE_F32) return KDA_ERR_INVALID_ARG;
    if (cp_mode < -1 || cp_mode > 1) return KDA_ERR_INVALID_ARG;
    if (segment_len < 0 || (segment_len % kChunk) != 0) return KDA_ERR_INVALID_ARG;
    if (!cu_seqlens) return KDA_ERR_INVALID_ARG;
    if (T > 0 && (!q || !k || !v || !g || !beta || !o)) return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(beta) ||
        !aligned16(o) || !aligned16(initial_state) || !aligned16(final_state) || !aligned16(workspace))
        return KDA_ERR_ALIGNMENT;
    if ((size_t)T * H * (dk > dv ? dk : dv) >= ((size_t)1 << 40)) return KDA_ERR_UNSUPPORTED_SHAPE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool bf = in_dtype == KDA_DTYPE_BF16;

    kda::ChunkArgs a = {};
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.o = o;
    a.T = T; a.H = H; a.dk = dk; a.dv = dv; a.scale = scale; a.g_min = g_min;
    a.status = status;
    a.cu_seqlens = cu_seqlens;
    if (ckpt_count > 0) {
        a.ckpt = ckpt;
        a.ckpt_every = ckpt_every;
        a.ckpt_count = ckpt_count;
    }

    CpLayout L = cp_layout(N, T, H, dk, dv, cp_mode, segment_len);
    // the two-kernel path when the workspace also holds its area
    SplitLayout SL;
    const size_t split_off = align256(L.total);
    bool split = bf && dk == 128 && dv == 128 && workspace && T > 0;
    if (split) {
        split = workspace_bytes > split_off;
        if (split) {
            SL = split_layout_fit(L.seg_len ? L.P_max : N, T, H, workspace_bytes - split_off, L.seg_len != 0);
            split = SL.piece >= 1;
        }
    }
    unsigned char *wsplit = split ? static_cast<unsigned char *>(workspace) + split_off : nullptr;
    if (L.seg_len == 0) {
        a.mode = kda::MODE_SEQ;
        a.cu_seqlens = cu_seqlens;
        a.S_init = initial_state;
        a.S_final = final_state;
        if (split) return cuda_status(run_split(a, N, wsplit, SL, true, false, st));
        return cuda_status(run_chunk(a, N, bf, st));
    }
    if (!workspace || workspace_bytes < L.total) return KDA_ERR_WORKSPACE;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    // one piece: the blobs written for the transitions (with Q~ and B) serve the replay too
    const bool one_piece = split && SL.piece >= SL.nslots;
    int32_t *count = reinterpret_cast<int32_t *>(ws + L.off_count);
    int32_t *table = reinterpret_cast<int32_t *>(ws + L.off_table);
    int32_t *first = reinterpret_cast<int32_t *>(ws + L.off_first);
    float *M = reinterpret_cast<float *>(ws + L.off_M);
    float *Nm = reinterpret_cast<float *>(ws + L.off_N);
    float *Sin = reinterpret_cast<float *>(ws + L.off_Sin);

    cudaError_t e = timed_launch(KDA_KERNEL_SEGMENT_TABLE, st, [&] {
        return kda::launch_segment_table(cu_seqlens, N, T, L.seg_len, L.P_max, table, first, count, status, st);
    });
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    // pass 1: transitions of every segment, independent of the incoming state
    a.mode = kda::MODE_TRANSITION;
    a.seg_table = table;
    a.seg_count = count;
    a.M_out = M;
    a.N_out = Nm;
    {
        kda::ChunkArgs at = a;  // transitions emit no checkpoints
        at.ckpt = nullptr;
        e = split ? run_split(at, L.P_max, wsplit, SL, one_piece, false, st) : run_chunk(at, L.P_max, bf, st);
    }
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    // pass 2: ordered scan per (sequence, head)
    kda::ComposeArgs c = {};
    c.M = M; c.Nm = Nm; c.S0 = initial_state; c.S_in = Sin; c.S_final = nullptr;
    c.first = first; c.P = 0; c.chains = N; c.H = H; c.dk = dk; c.dv = dv;
    e = timed_launch(KDA_KERNEL_SEGMENT_COMPOSE, st, [&] { return kda::launch_compose(c, st); });
    if (e != cudaSuccess) return KDA_ERR_CUDA;
    // pass 3: replay every segment from its exact initial state
    a.mode = kda::MODE_REPLAY;
    a.S_in = Sin;
    a.S_final = final_state;
    a.M_out = a.N_out = nullptr;
    if (split) return cuda_status(run_split(a, L.P_max, wsplit, SL, true, one_piece, st));
    return cuda_status(run_chunk(a, L.P_max, bf, st));
}

}  // namespace

int kda_chunk_fwd(const void *q, const void *k, const void *v, const float *g, const float *beta,
                  const int32_t *cu_seqlens, int N, int T, int H, int dk, int dv,
                  const float *initial_state, float *final_state, void *o, float scale, float g_min,
                  int in_dtype, int cp_mode, int segment_len, void *workspace, size_t workspace_bytes,
                  uint32_t *status, void *stream) {
    return chunk_fwd_impl(q, k, v, g, beta, cu_seqlens, N, T, H, dk, dv, initial_state, final_state, o, scale,
                          g_min, in_dtype, cp_mode, segment_len, workspace, workspace_bytes, 0, 0, nullptr,
                          status, stream);
}

int kda_chunk_fwd_ckpt(const void *q, const void *k, const void *v, const float *g, const float *beta,
                       const int32_t *cu_seqlens, int N, int T, int H, int dk, int dv,
                       const float *initial_state, float *final_state, void *o, float scale, float g_min,
                       int in_dtype, int cp_mode, int segment_len, void *workspace, size_t workspace_bytes,
                       int ckpt_every, int ckpt_count, float *ckpt, uint32_t *status, void *stream) {
    if (ckpt_every <= 0 || (ckpt_every % kChunk) != 0 || ckpt_count < 0) return KDA_ERR_INVALID_ARG;
    if (ckpt_count > 0 && !ckpt) return KDA_ERR_INVALID_ARG;
    if (!aligned16(ckpt)) return KDA_ERR_ALIGNMENT;
    return chunk_fwd_impl(q, k, v, g, beta, cu_seqlens, N, T, H, dk, dv, initial_state, final_state, o, scale,
                          g_min, in_dtype, cp_mode, segment_len, workspace, workspace_bytes, ckpt_every,
                          ckpt_count, ckpt, status, stream);
}

int kda_segment_transition(const void *k, const void *v, const float *g, const float *beta, int T, int H,
                           int dk, int dv, int segment_len, float *M, float *Nmat, float g_min,
                           int in_dtype, void *stream) {
    if (T < 0 || H < 1 || segment_len <= 0 || (segment_len % kChunk) != 0) return KDA_ERR_INVALID_ARG;
    if (!dim_ok(dk) || !dim_ok(dv)) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (in_dtype != KDA_DTYPE_BF16 && in_dtype != KDA_DTYPE_F32) return KDA_ERR_INVALID_ARG;
    if (T > 0 && (!k || !v || !g || !beta || !M || !Nmat)) return KDA_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(beta) || !aligned16(M) ||
        !aligned16(Nmat))
        return KDA_ERR_ALIGNMENT;
    if (T == 0) return KDA_OK;
    kda::ChunkArgs a = {};
    a.q = nullptr; a.k = k; a.v = v; a.g = g; a.beta = beta; a.o = nullptr;
    a.T = T; a.H = H; a.dk = dk; a.dv = dv; a.scale = 1.f; a.g_min = g_min;
    a.mode = kda::MODE_TRANSITION;
    a.seg_table = nullptr;
    a.seg_len = segment_len;
    a.M_out = M;
    a.N_out = Nmat;
    const int P = (T + segment_len - 1) / segment_len;
    return cuda_status(run_chunk(a, P, in_dtype == KDA_DTYPE_BF16, static_cast<cudaStream_t>(stream)));
}

int kda_segment_compose(const float *M, const float *Nmat, const float *S0, float *S_in, float *S_final,
                        int P, int H, int dk, int dv, void *stream) {
    if (P < 0 || H < 1) return KDA_ERR_INVALID_ARG;
    if (!dim_ok(dk) || !dim_ok(dv)) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (P > 0 && (!M || !Nmat)) return KDA_ERR_INVALID_ARG;
    if (!aligned16(M) || !aligned16(Nmat) || !aligned16(S0) || !aligned16(S_in) || !aligned16(S_final))
        return KDA_ERR_ALIGNMENT;
    kda::ComposeArgs c = {};
    c.M = M; c.Nm = Nmat; c.S0 = S0; c.S_in = S_in; c.S_final = S_final;
    c.first = nullptr; c.P = P; c.chains = 1; c.H = H; c.dk = dk; c.dv = dv;
    return cuda_status(kda::launch_compose(c, static_cast<cudaStream_t>(stream)));
}

int kda_decode_verify_replay(void *state, void *conv_tail, const float *conv_w, const void *cached_qkv,
                             const void *cached_g, const void *cached_beta, const int32_t *accepted_len,
                             const void *new_qkv, const void *new_g, const void *new_beta,
                             const float *out_norm_w, void *o, int R, int H, int dk, int dv, int W, int Wd,
                             float scale, float g_min, float eps_in, float eps_out, int conv_act,
                             uint32_t *status, void *stream) {
    return kda_decode_verify_replay_ragged(state, conv_tail, conv_w, cached_qkv, cached_g, cached_beta,
                                           accepted_len, nullptr, new_qkv, new_g, new_beta, out_norm_w, o, R,
                                           H, dk, dv, W, Wd, scale, g_min, eps_in, eps_out, conv_act, status,
                                           stream);
}

int kda_decode_verify_replay_ragged(void *state, void *conv_tail, const float *conv_w, const void *cached_qkv,
                                    const void *cached_g, const void *cached_beta, const int32_t *accepted_len,
                                    const int32_t *draft_len, const void *new_qkv, const void *new_g,
                                    const void *new_beta, const float *out_norm_w, void *o, int R, int H,
                                    int dk, int dv, int W, int Wd, float scale, float g_min, float eps_in,
                                    float eps_out, int conv_act, uint32_t *status, void *stream) {
    if (R < 0 || H < 1 || W < 1 || W > 4 || Wd < 0 || Wd > 7) return KDA_ERR_INVALID_ARG;
    if (conv_act != KDA_CONV_NONE && conv_act != KDA_CONV_SILU) return KDA_ERR_INVALID_ARG;
    if (!(dk == dv && dim_ok(dk))) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (R > 0 && (!state || !conv_w || !accepted_len || !new_qkv || !new_g || !new_beta || !out_norm_w ||
                  !o || (W > 1 && !conv_tail) || (Wd > 0 && (!cached_qkv || !cached_g || !cached_beta))))
        return KDA_ERR_INVALID_ARG;
    if (!aligned16(state) || !aligned16(conv_tail) || !aligned16(conv_w) || !aligned16(cached_qkv) ||
        !aligned16(cached_g) || !aligned16(new_qkv) || !aligned16(new_g) || !aligned16(o) ||
        !aligned16(out_norm_w))
        return KDA_ERR_ALIGNMENT;
    if ((size_t)R * H >= ((size_t)1 << 31)) return KDA_ERR_UNSUPPORTED_SHAPE;
    kda::VerifyArgs a = {};
    a.state = state; a.tail = conv_tail; a.conv_w = conv_w;
    a.cached_qkv = cached_qkv; a.cached_g = cached_g; a.cached_b = cached_beta;
    a.accepted = accepted_len;
    a.draft_len = draft_len;
    a.new_qkv = new_qkv; a.new_g = new_g; a.new_b = new_beta;
    a.out_w = out_norm_w; a.o = o;
    a.R = R; a.H = H; a.dk = dk; a.dv = dv; a.W = W; a.Wd = Wd;
    a.scale = scale; a.g_min = g_min; a.eps_in = eps_in; a.eps_out = eps_out; a.conv_act = conv_act;
    a.status = status;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return cuda_status(timed_launch(KDA_KERNEL_VERIFY, st, [&] { return kda::launch_verify(a, st); }));
}

namespace {
// Workspace of the tensor-core backward (d = 128, bf16): per (slot, head) the
// forward pass's operand blob, T and M^T (f32), the walk's S^T and U^T tiles
// and the reverse walk's dS'^T and dU'^T tiles; the slot list and the item
// counters in front.
struct BwdTcLayout {
    size_t nslots, off_list, off_claim, off_carry, carry_stride, off_blob, off_aux, off_s, off_u, off_ds, off_du,
        total;
};
BwdTcLayout bwd_tc_layout(int N, int T, int H) {  // N units: sequences, or segments
    BwdTcLayout L;
    L.nslots = (size_t)T / kChunk + N;
    const size_t sh = L.nslots * H;
    size_t off = 0;
    L.off_list = off;
    off += align256(L.nslots * sizeof(int2));
    L.off_claim = off;  // one item counter per piece of the forward pass, one for the chunk kernel
    off += 256;
    L.off_carry = off;  // two states per head for a sequence cut between pieces
    L.carry_stride = (size_t)H * 128 * 128;
    off += align256(2 * L.carry_stride * 4);
    L.off_blob = off;
    off += align256(sh * kda::kChunkBlobBytes);
    L.off_aux = off;
    off += align256(sh * 32768);
    L.off_s = off;
    off += align256(sh * 32768);
    L.off_u = off;
    off += align256(sh * 16384);
    L.off_ds = off;
    off += align256(sh * 32768);
    L.off_du = off;
    off += align256(sh * 16384);
    L.total = off;
    return L;
}
}  // namespace

namespace {
kda::ChunkArgs bwd_tc_fwd_args(const void *q, const void *k, const void *v, const float *g, const float *beta,
                               const int32_t *cu_seqlens, int T, int H, const float *S0, float *S_final, void *o,
                               float scale, float g_min, uint32_t *status) {
    kda::ChunkArgs fa = {};
    fa.q = q; fa.k = k; fa.v = v; fa.g = g; fa.beta = beta; fa.o = o;
    fa.T = T; fa.H = H; fa.dk = 128; fa.dv = 128; fa.scale = scale; fa.g_min = g_min;
    fa.mode = kda::MODE_SEQ; fa.cu_seqlens = cu_seqlens; fa.S_init = S0; fa.S_final = S_final; fa.status = status;
    return fa;
}

kda::BwdTcArgs bwd_tc_args(const void *q, const void *k, const void *v, const float *g, const float *beta,
                           const int32_t *cu_seqlens, int N, int T, int H, const void *dout, const float *dS_final,
                           float *dq, float *dk, float *dv, float *dg, float *dbeta, float *dS0, float scale,
                           float g_min, unsigned char *ws, uint32_t *status, int layout_units = -1) {
    // the workspace is laid out for N sequences, or for layout_units segments
    const BwdTcLayout L = bwd_tc_layout(layout_units < 0 ? N : layout_units, T, H);
    kda::BwdTcArgs b = {};
    b.q = q; b.k = k; b.v = v; b.dout = dout; b.g = g; b.beta = beta; b.cu_seqlens = cu_seqlens;
    b.N = N; b.T = T; b.H = H; b.scale = scale; b.g_min = g_min; b.dS_final = dS_final;
    b.dq = dq; b.dk = dk; b.dv = dv; b.dg = dg; b.dbeta = dbeta; b.dS0 = dS0;
    b.list = reinterpret_cast<const int2 *>(ws + L.off_list);
    b.blob = ws + L.off_blob;
    b.aux = reinterpret_cast<const float *>(ws + L.off_aux);
    b.save_s = ws + L.off_s; b.save_u = ws + L.off_u; b.save_ds = ws + L.off_ds; b.save_du = ws + L.off_du;
    b.status = status;
    return b;
}

int bwd_tc_pieces(int N, int T, int H) { return pipe_wanted(N, T, H, false) ? kPipePieces : 1; }

// The forward pass of the tensor-core backward, in the prefill's pieces: the
// chunk-local launch of piece p + 1 a programmatic dependent of the walk of
// piece p (it reads nothing the walk writes, and every piece keeps its own
// blobs, T and M for the reverse walk and the chunk kernel); the walks keep
// their state and U tiles, and write o and S_final when fa has them.
cudaError_t bwd_tc_forward(const kda::ChunkArgs &fa, int N, int T, int H, unsigned char *ws, cudaStream_t st) {
    const BwdTcLayout L = bwd_tc_layout(N, T, H);
    const int nslots = (int)L.nslots, P = bwd_tc_pieces(N, T, H), piece = (nslots + P - 1) / P;
    int2 *list = reinterpret_cast<int2 *>(ws + L.off_list);
    int *claim = reinterpret_cast<int *>(ws + L.off_claim);
    unsigned char *blob = ws + L.off_blob;
    float *aux = reinterpret_cast<float *>(ws + L.off_aux);
    float *carry = reinterpret_cast<float *>(ws + L.off_carry);
    cudaError_t e = cudaMemsetAsync(claim, 0, (size_t)P * sizeof(int), st);
    if (e == cudaSuccess)
        e = timed_launch(KDA_KERNEL_CHUNK_LIST, st, [&] { return kda::launch_chunk_list(fa, N, nslots, list, st); });
    for (int pc = 0; e == cudaSuccess && T > 0 && pc < P; ++pc) {
        const int s0 = pc * piece, s1 = s0 + piece < nslots ? s0 + piece : nslots;
        if (s0 >= s1) break;
        unsigned char *pb = blob + (size_t)s0 * H * kda::kChunkBlobBytes;
        e = timed_launch(KDA_KERNEL_CHUNK_PREP, st, [&] {
            return kda::launch_chunk_prep(fa, list, s0, s1, pb, true, claim + pc, pc > 0, st, aux + (size_t)s0 * H * 8192);
        });
        if (e == cudaSuccess)
            e = timed_launch(KDA_KERNEL_CHUNK_WALK, st, [&] {
                return kda::launch_chunk_walk(fa, N, pb, s0, s1, carry + (size_t)(pc & 1) * L.carry_stride,
                                              carry + (size_t)((pc + 1) & 1) * L.carry_stride, st, ws + L.off_s,
                                              ws + L.off_u);
            });
    }
    if (e == cudaSuccess && T == 0 && fa.S_final && N > 0) {  // no chunk: the final states are the initial ones
        const size_t bytes = (size_t)N * H * 128 * 128 * 4;
        e = fa.S_init ? cudaMemcpyAsync(fa.S_final, fa.S_init, bytes, cudaMemcpyDeviceToDevice, st)
                      : cudaMemsetAsync(fa.S_final, 0, bytes, st);
    }
    return e;
}

// The reverse pass over what bwd_tc_forward kept, in the same pieces, newest
// first: the chunk gradients of piece p (which need its reverse walk
// complete) run as a programmatic dependent of the reverse walk of the piece
// before it in slot order, on the SMs that walk leaves free.
cudaError_t bwd_tc_reverse(const kda::BwdTcArgs &b, int N, int T, int H, unsigned char *ws, cudaStream_t st) {
    const BwdTcLayout L = bwd_tc_layout(N, T, H);
    const int nslots = (int)L.nslots, P = bwd_tc_pieces(N, T, H), piece = (nslots + P - 1) / P;
    int *claim = reinterpret_cast<int *>(ws + L.off_claim) + P;
    float *carry = reinterpret_cast<float *>(ws + L.off_carry);
    cudaError_t e = cudaMemsetAsync(claim, 0, (size_t)P * sizeof(int), st);
    auto rpiece = [&](int r, int &s0, int &s1) {  // r-th piece of the reverse pass
        const int pc = P - 1 - r;
        s0 = pc * piece;
        s1 = s0 + piece < nslots ? s0 + piece : nslots;
    };
    for (int r = 0; e == cudaSuccess && r <= P; ++r) {
        int s0 = 0, s1 = 0;
        if (r < P) {
            rpiece(r, s0, s1);
            if (T == 0) {
                s0 = 0;
                s1 = nslots;
            }
            e = timed_launch(KDA_KERNEL_BWD_WALK, st, [&] {
                return kda::launch_bwd_walk(b, s0, s1, carry + (size_t)(r & 1) * L.carry_stride,
                                            carry + (size_t)((r + 1) & 1) * L.carry_stride, st);
            });
            if (T == 0) break;
        }
        if (e == cudaSuccess && r > 0) {
            int c0 = 0, c1 = 0;
            rpiece(r - 1, c0, c1);
            e = timed_launch(KDA_KERNEL_BWD_CHUNK, st,
                             [&] { return kda::launch_bwd_chunk(b, c0, c1, claim + (r - 1), r < P, st); });
        }
    }
    return e;
}

// Shape, pointer and workspace checks of the tensor-core training pair.
int train_pair_check(int N, int T, int H, int dk, int dv, int in_dtype, const int32_t *cu_seqlens, void *saved,
                     size_t saved_bytes) {
    if (N < 1 || T < 0 || H < 1 || !cu_seqlens) return KDA_ERR_INVALID_ARG;
    if (dk != 128 || dv != 128 || in_dtype != KDA_DTYPE_BF16) return KDA_ERR_UNSUPPORTED_SHAPE;
    if ((size_t)T * H * dk >= ((size_t)1 << 40)) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(saved)) return KDA_ERR_ALIGNMENT;
    if (!saved || saved_bytes < bwd_tc_layout(N, T, H).total) return KDA_ERR_WORKSPACE;
    return KDA_OK;
}
}  // namespace

size_t kda_chunk_bwd_workspace_size(int N, int T, int H, int dk, int dv) {
    if (N < 1 || T < 0 || H < 1 || dk != dv || !dim_ok(dk)) return 0;
    const size_t DD = (size_t)dk * dv * 4;
    const size_t units = (size_t)N * H, slots = units < (size_t)kda::kBwdMaxCtas ? units : (size_t)kda::kBwdMaxCtas;
    const size_t parts = slots * (size_t)(dk / 32) * 2 * kda::chunk_bwd_partial_floats(dk) * 4;
    const size_t cores = align256((size_t)(T / kChunk + N) * H * DD) + align256(slots * kChunk * DD) +
                         align256(parts) + align256((size_t)T * H * dk * 4);
    if (dk != 128) return cores;
    const size_t tc = bwd_tc_layout(N, T, H).total;  // bf16 inputs take the tensor-core form
    return tc > cores ? tc : cores;
}

int kda_chunk_bwd(const void *q, const void *k, const void *v, const float *g, const float *beta,
                  const int32_t *cu_seqlens, int N, int T, int H, int dk, int dv, const float *initial_state,
                  const void *dout, const float *dS_final, float *dq, float *dk_, float *dv_, float *dg,
                  float *dbeta, float *dS0, float scale, float g_min, int in_dtype, void *workspace,
                  size_t workspace_bytes, uint32_t *status, void *stream) {
    if (N < 1 || T < 0 || H < 1 || !cu_seqlens) return KDA_ERR_INVALID_ARG;
    if (dk != dv || !dim_ok(dk)) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (in_dtype != KDA_DTYPE_BF16 && in_dtype != KDA_DTYPE_F32) return KDA_ERR_INVALID_ARG;
    if (T > 0 && (!q || !k || !v || !g || !beta || !dout || !dq || !dk_ || !dv_ || !dg || !dbeta))
        return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(dout) ||
        !aligned16(initial_state) || !aligned16(dS_final) || !aligned16(dS0) || !aligned16(workspace))
        return KDA_ERR_ALIGNMENT;
    if ((size_t)T * H * dk >= ((size_t)1 << 40)) return KDA_ERR_UNSUPPORTED_SHAPE;
    const size_t need = kda_chunk_bwd_workspace_size(N, T, H, dk, dv);
    if (!workspace || workspace_bytes < need) return KDA_ERR_WORKSPACE;
    const size_t DD = (size_t)dk * dv * 4;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (dk == 128 && in_dtype == KDA_DTYPE_BF16) {
        // the chunk (WY) form on the tensor cores: forward pass keeping its
        // operands, reverse state walk, chunk gradients
        kda::ChunkArgs fa = bwd_tc_fwd_args(q, k, v, g, beta, cu_seqlens, T, H, initial_state, nullptr, nullptr, scale,
                                            g_min, status);
        cudaError_t e = bwd_tc_forward(fa, N, T, H, ws, st);
        if (e == cudaSuccess)
            e = bwd_tc_reverse(bwd_tc_args(q, k, v, g, beta, cu_seqlens, N, T, H, dout, dS_final, dq, dk_, dv_, dg,
                                           dbeta, dS0, scale, g_min, ws, status),
                               N, T, H, ws, st);
        return cuda_status(e);
    }
    kda::BwdArgs a = {};
    a.q = q; a.k = k; a.v = v; a.dout = dout; a.g = g; a.beta = beta; a.cu_seqlens = cu_seqlens;
    a.S0 = initial_state; a.dS_final = dS_final;
    a.dq = dq; a.dk = dk_; a.dv = dv_; a.dg = dg; a.dbeta = dbeta; a.dS0 = dS0;
    a.ckpt = reinterpret_cast<float *>(ws);
    const size_t units = (size_t)N * H, slots = units < (size_t)kda::kBwdMaxCtas ? units : (size_t)kda::kBwdMaxCtas;
    const size_t off_scr = align256((size_t)(T / kChunk + N) * H * DD);
    a.scratch = reinterpret_cast<float *>(ws + off_scr);
    const size_t off_par = off_scr + align256(slots * kChunk * DD);
    a.partials = reinterpret_cast<float *>(ws + off_par);
    a.wbuf = reinterpret_cast<float *>(
        ws + off_par + align256(slots * (size_t)(dk / 32) * 2 * kda::chunk_bwd_partial_floats(dk) * 4));
    a.N = N; a.T = T; a.H = H; a.scale = scale; a.g_min = g_min; a.status = status;
    return cuda_status(timed_launch(KDA_KERNEL_CHUNK_BWD, st,
                                    [&] { return kda::launch_chunk_bwd(a, dk, in_dtype == KDA_DTYPE_BF16, st); }));
}

int kda_chunk_fwd_train(const void *q, const void *k, const void *v, const float *g, const float *beta,
                        const int32_t *cu_seqlens, int N, int T, int H, int dk, int dv, const float *initial_state,
                        float *final_state, void *o, float scale, float g_min, int in_dtype, void *saved,
                        size_t saved_bytes, uint32_t *status, void *stream) {
    int rc = train_pair_check(N, T, H, dk, dv, in_dtype, cu_seqlens, saved, saved_bytes);
    if (rc != KDA_OK) return rc;
    if (T > 0 && (!q || !k || !v || !g || !beta || !o)) return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(o) ||
        !aligned16(initial_state) || !aligned16(final_state))
        return KDA_ERR_ALIGNMENT;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned char *ws = static_cast<unsigned char *>(saved);
    return cuda_status(bwd_tc_forward(bwd_tc_fwd_args(q, k, v, g, beta, cu_seqlens, T, H, initial_state, final_state,
                                                      o, scale, g_min, status),
                                      N, T, H, ws, st));
}

int kda_chunk_bwd_saved(const void *q, const void *k, const void *v, const float *g, const float *beta,
                        const int32_t *cu_seqlens, int N, int T, int H, int dk, int dv, const void *dout,
                        const float *dS_final, float *dq, float *dk_, float *dv_, float *dg, float *dbeta,
                        float *dS0, float scale, float g_min, int in_dtype, void *saved, size_t saved_bytes,
                        uint32_t *status, void *stream) {
    int rc = train_pair_check(N, T, H, dk, dv, in_dtype, cu_seqlens, saved, saved_bytes);
    if (rc != KDA_OK) return rc;
    if (T > 0 && (!q || !k || !v || !g || !beta || !dout || !dq || !dk_ || !dv_ || !dg || !dbeta))
        return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(dout) ||
        !aligned16(dS_final) || !aligned16(dS0))
        return KDA_ERR_ALIGNMENT;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned char *ws = static_cast<unsigned char *>(saved);
    return cuda_status(bwd_tc_reverse(bwd_tc_args(q, k, v, g, beta, cu_seqlens, N, T, H, dout, dS_final, dq, dk_, dv_,
                                                  dg, dbeta, dS0, scale, g_min, ws, status),
                                      N, T, H, ws, st));
}

namespace {
// Workspace of the context-parallel backward: the forward's CP area (segment
// table, transitions, segment states), the tensor-core layout over the
// segments' slots, then r and dS_end per (segment, head).
struct BwdCpLayout {
    CpLayout cp;
    size_t off_tc = 0, off_r = 0, off_end = 0, total = 0;
};
BwdCpLayout bwd_cp_layout(int N, int T, int H, int cp_mode, int segment_len) {
    BwdCpLayout B;
    B.cp = cp_layout(N, T, H, 128, 128, cp_mode, segment_len);
    if (B.cp.seg_len == 0) return B;
    size_t o = align256(B.cp.total);
    B.off_tc = o;
    o += align256(bwd_tc_layout(B.cp.P_max, T, H).total);
    const size_t st = (size_t)B.cp.P_max * H * 128 * 128 * 4;
    B.off_r = o;
    o += align256(st);
    B.off_end = o;
    o += align256(st);
    B.total = o;
    return B;
}
}  // namespace

size_t kda_chunk_bwd_cp_workspace_size(int N, int T, int H, int dk, int dv, int cp_mode, int segment_len) {
    const size_t base = kda_chunk_bwd_workspace_size(N, T, H, dk, dv);
    if (base == 0 || dk != 128 || cp_mode == KDA_CP_OFF) return base;
    if (cp_mode != KDA_CP_ON && cp_mode != KDA_CP_AUTO) return 0;
    const BwdCpLayout B = bwd_cp_layout(N, T, H, cp_mode, segment_len);
    return B.total > base ? B.total : base;
}

namespace {
// Pointers into the context-parallel backward's workspace.
struct BwdCpPtrs {
    int32_t *count, *table, *first;
    float *M, *Nm, *Sin, *r, *dend;
    unsigned char *tw;  // the tensor-core layout over the segments' slots
    int Pm, nslots;
};
BwdCpPtrs bwd_cp_ptrs(const BwdCpLayout &B, int T, int H, unsigned char *ws) {
    const CpLayout &C = B.cp;
    BwdCpPtrs p;
    p.count = reinterpret_cast<int32_t *>(ws + C.off_count);
    p.table = reinterpret_cast<int32_t *>(ws + C.off_table);
    p.first = reinterpret_cast<int32_t *>(ws + C.off_first);
    p.M = reinterpret_cast<float *>(ws + C.off_M);
    p.Nm = reinterpret_cast<float *>(ws + C.off_N);
    p.Sin = reinterpret_cast<float *>(ws + C.off_Sin);
    p.r = reinterpret_cast<float *>(ws + B.off_r);
    p.dend = reinterpret_cast<float *>(ws + B.off_end);
    p.tw = ws + B.off_tc;
    p.Pm = C.P_max;
    p.nslots = (int)bwd_tc_layout(C.P_max, T, H).nslots;
    return p;
}

// The forward pass as the CP prefill runs it, keeping what the reverse pass
// needs: segment table, every chunk's blob (with T and M^T), the transitions
// of every segment, their ordered composition, and the replay from each
// segment's exact start keeping its state and U tiles (and writing o and the
// final states when a has them).
cudaError_t bwd_cp_forward(kda::ChunkArgs a, int N, int T, int H, const BwdCpLayout &B, unsigned char *ws,
                           cudaStream_t st) {
    const BwdCpPtrs w = bwd_cp_ptrs(B, T, H, ws);
    const BwdTcLayout L = bwd_tc_layout(w.Pm, T, H);
    int2 *list = reinterpret_cast<int2 *>(w.tw + L.off_list);
    int *claim = reinterpret_cast<int *>(w.tw + L.off_claim);
    unsigned char *blob = w.tw + L.off_blob;
    float *aux = reinterpret_cast<float *>(w.tw + L.off_aux);
    a.seg_len = B.cp.seg_len;
    a.seg_table = w.table;
    a.seg_count = w.count;
    cudaError_t e = timed_launch(KDA_KERNEL_SEGMENT_TABLE, st, [&] {
        return kda::launch_segment_table(a.cu_seqlens, N, T, B.cp.seg_len, w.Pm, w.table, w.first, w.count,
                                         a.status, st);
    });
    if (e == cudaSuccess) e = cudaMemsetAsync(claim, 0, 2 * sizeof(int), st);
    kda::ChunkArgs ar = a;
    ar.mode = kda::MODE_REPLAY;
    ar.S_in = w.Sin;
    if (e == cudaSuccess)
        e = timed_launch(KDA_KERNEL_CHUNK_LIST, st,
                         [&] { return kda::launch_chunk_list(ar, w.Pm, w.nslots, list, st); });
    if (e == cudaSuccess)
        e = timed_launch(KDA_KERNEL_CHUNK_PREP, st, [&] {
            return kda::launch_chunk_prep(ar, list, 0, w.nslots, blob, true, claim, false, st, aux);
        });
    kda::ChunkArgs at = a;
    at.mode = kda::MODE_TRANSITION;
    at.o = nullptr;
    at.S_final = nullptr;
    at.M_out = w.M;
    at.N_out = w.Nm;
    if (e == cudaSuccess)
        e = timed_launch(KDA_KERNEL_CHUNK_WALK, st, [&] {
            return kda::launch_chunk_walk(at, w.Pm, blob, 0, w.nslots, nullptr, nullptr, st);
        });
    kda::ComposeArgs c = {};
    c.M = w.M; c.Nm = w.Nm; c.S0 = a.S_init; c.S_in = w.Sin; c.S_final = nullptr;
    c.first = w.first; c.P = 0; c.chains = N; c.H = H; c.dk = 128; c.dv = 128;
    if (e == cudaSuccess) e = timed_launch(KDA_KERNEL_SEGMENT_COMPOSE, st, [&] { return kda::launch_compose(c, st); });
    if (e == cudaSuccess)
        e = timed_launch(KDA_KERNEL_CHUNK_WALK, st, [&] {
            return kda::launch_chunk_walk(ar, w.Pm, blob, 0, w.nslots, nullptr, nullptr, st, w.tw + L.off_s,
                                          w.tw + L.off_u);
        });
    return e;
}

// The reverse pass over what bwd_cp_forward kept: every segment walked back
// from zero (r), the state gradient scanned over the segments last to first,
// every segment walked back again from its exact end gradient keeping its
// tiles, then the chunk gradients.
cudaError_t bwd_cp_reverse(kda::BwdTcArgs b, int N, int T, int H, const BwdCpLayout &B, unsigned char *ws,
                           float scale, cudaStream_t st) {
    const BwdCpPtrs w = bwd_cp_ptrs(B, T, H, ws);
    const BwdTcLayout L = bwd_tc_layout(w.Pm, T, H);
    int *claim = reinterpret_cast<int *>(w.tw + L.off_claim);
    cudaError_t e = cudaMemsetAsync(claim + 1, 0, sizeof(int), st);
    kda::BwdSegments sg = {w.table, w.count, w.Pm, nullptr, w.r, false};
    if (e == cudaSuccess)
        e = timed_launch(KDA_KERNEL_BWD_WALK, st, [&] {
            return kda::launch_bwd_walk(b, 0, w.nslots, nullptr, nullptr, st, &sg);
        });
    if (e == cudaSuccess)
        e = timed_launch(KDA_KERNEL_BWD_COMPOSE, st, [&] {
            return kda::launch_bwd_compose(w.M, w.r, w.first, b.cu_seqlens, b.dS_final, w.dend, b.dS0, N, H, scale,
                                           st);
        });
    kda::BwdSegments sg2 = {w.table, w.count, w.Pm, w.dend, nullptr, true};
    if (e == cudaSuccess)
        e = timed_launch(KDA_KERNEL_BWD_WALK, st, [&] {
            return kda::launch_bwd_walk(b, 0, w.nslots, nullptr, nullptr, st, &sg2);
        });
    if (e == cudaSuccess)
        e = timed_launch(KDA_KERNEL_BWD_CHUNK, st,
                         [&] { return kda::launch_bwd_chunk(b, 0, w.nslots, claim + 1, false, st); });
    return e;
}

// The CP backward's layout when the call is cut into segments (bf16,
// d = 128, T > 0), else an empty layout (seg_len 0).
BwdCpLayout bwd_cp_plan(int N, int T, int H, int dk, int dv, int in_dtype, int cp_mode, int segment_len) {
    if (dk == 128 && dv == 128 && in_dtype == KDA_DTYPE_BF16 && N >= 1 && H >= 1 && T > 0)
        return bwd_cp_layout(N, T, H, cp_mode, segment_len);
    return BwdCpLayout();
}

int bwd_cp_check_args(int cp_mode, int segment_len) {
    if (cp_mode != KDA_CP_OFF && cp_mode != KDA_CP_ON && cp_mode != KDA_CP_AUTO) return KDA_ERR_INVALID_ARG;
    if (segment_len < 0 || segment_len % kChunk != 0) return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}
}  // namespace

int kda_chunk_bwd_cp(const void *q, const void *k, const void *v, const float *g, const float *beta,
                     const int32_t *cu_seqlens, int N, int T, int H, int dk, int dv, const float *initial_state,
                     const void *dout, const float *dS_final, float *dq, float *dk_, float *dv_, float *dg,
                     float *dbeta, float *dS0, float scale, float g_min, int in_dtype, int cp_mode, int segment_len,
                     void *workspace, size_t workspace_bytes, uint32_t *status, void *stream) {
    int rc = bwd_cp_check_args(cp_mode, segment_len);
    if (rc != KDA_OK) return rc;
    const BwdCpLayout B = bwd_cp_plan(N, T, H, dk, dv, in_dtype, cp_mode, segment_len);
    if (B.cp.seg_len == 0)  // no segments for this call: the sequence form
        return kda_chunk_bwd(q, k, v, g, beta, cu_seqlens, N, T, H, dk, dv, initial_state, dout, dS_final, dq, dk_,
                             dv_, dg, dbeta, dS0, scale, g_min, in_dtype, workspace, workspace_bytes, status, stream);
    if (!cu_seqlens || !q || !k || !v || !g || !beta || !dout || !dq || !dk_ || !dv_ || !dg || !dbeta)
        return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(dout) ||
        !aligned16(initial_state) || !aligned16(dS_final) || !aligned16(dS0) || !aligned16(workspace))
        return KDA_ERR_ALIGNMENT;
    if ((size_t)T * H * dk >= ((size_t)1 << 40)) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (!workspace || workspace_bytes < B.total) return KDA_ERR_WORKSPACE;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = bwd_cp_forward(bwd_tc_fwd_args(q, k, v, g, beta, cu_seqlens, T, H, initial_state, nullptr,
                                                   nullptr, scale, g_min, status),
                                   N, T, H, B, ws, st);
    if (e == cudaSuccess)
        e = bwd_cp_reverse(bwd_tc_args(q, k, v, g, beta, cu_seqlens, N, T, H, dout, dS_final, dq, dk_, dv_, dg,
                                       dbeta, dS0, scale, g_min, ws + B.off_tc, status, B.cp.P_max),
                           N, T, H, B, ws, scale, st);
    return cuda_status(e);
}

int kda_chunk_fwd_train_cp(const void *q, const void *k, const void *v, const float *g, const float *beta,
                           const int32_t *cu_seqlens, int N, int T, int H, int dk, int dv,
                           const float *initial_state, float *final_state, void *o, float scale, float g_min,
                           int in_dtype, int cp_mode, int segment_len, void *saved, size_t saved_bytes,
                           uint32_t *status, void *stream) {
    int rc = bwd_cp_check_args(cp_mode, segment_len);
    if (rc != KDA_OK) return rc;
    const BwdCpLayout B = bwd_cp_plan(N, T, H, dk, dv, in_dtype, cp_mode, segment_len);
    if (B.cp.seg_len == 0)
        return kda_chunk_fwd_train(q, k, v, g, beta, cu_seqlens, N, T, H, dk, dv, initial_state, final_state, o,
                                   scale, g_min, in_dtype, saved, saved_bytes, status, stream);
    if (!cu_seqlens || !q || !k || !v || !g || !beta || !o) return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(o) ||
        !aligned16(initial_state) || !aligned16(final_state) || !aligned16(saved))
        return KDA_ERR_ALIGNMENT;
    if ((size_t)T * H * dk >= ((size_t)1 << 40)) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (!saved || saved_bytes < B.total) return KDA_ERR_WORKSPACE;
    return cuda_status(bwd_cp_forward(bwd_tc_fwd_args(q, k, v, g, beta, cu_seqlens, T, H, initial_state,
                                                      final_state, o, scale, g_min, status),
                                      N, T, H, B, static_cast<unsigned char *>(saved),
                                      static_cast<cudaStream_t>(stream)));
}

int kda_chunk_bwd_saved_cp(const void *q, const void *k, const void *v, const float *g, const float *beta,
                           const int32_t *cu_seqlens, int N, int T, int H, int dk, int dv, const void *dout,
                           const float *dS_final, float *dq, float *dk_, float *dv_, float *dg, float *dbeta,
                           float *dS0, float scale, float g_min, int in_dtype, int cp_mode, int segment_len,
                           void *saved, size_t saved_bytes, uint32_t *status, void *stream) {
    int rc = bwd_cp_check_args(cp_mode, segment_len);
    if (rc != KDA_OK) return rc;
    const BwdCpLayout B = bwd_cp_plan(N, T, H, dk, dv, in_dtype, cp_mode, segment_len);
    if (B.cp.seg_len == 0)
        return kda_chunk_bwd_saved(q, k, v, g, beta, cu_seqlens, N, T, H, dk, dv, dout, dS_final, dq, dk_, dv_, dg,
                                   dbeta, dS0, scale, g_min, in_dtype, saved, saved_bytes, status, stream);
    if (!cu_seqlens || !q || !k || !v || !g || !beta || !dout || !dq || !dk_ || !dv_ || !dg || !dbeta)
        return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(dout) ||
        !aligned16(dS_final) || !aligned16(dS0) || !aligned16(saved))
        return KDA_ERR_ALIGNMENT;
    if ((size_t)T * H * dk >= ((size_t)1 << 40)) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (!saved || saved_bytes < B.total) return KDA_ERR_WORKSPACE;
    unsigned char *ws = static_cast<unsigned char *>(saved);
    return cuda_status(bwd_cp_reverse(bwd_tc_args(q, k, v, g, beta, cu_seqlens, N, T, H, dout, dS_final, dq, dk_,
                                                  dv_, dg, dbeta, dS0, scale, g_min, ws + B.off_tc, status,
                                                  B.cp.P_max),
                                      N, T, H, B, ws, scale, static_cast<cudaStream_t>(stream)));
}

size_t kda_chunk_fwd_host_workspace_size(int N, int T, int H, int dk, int dv, int in_dtype, int pieces) {
    if (N < 1 || T < 0 || H < 1 || !dim_ok(dk) || !dim_ok(dv)) return 0;
    if (in_dtype != KDA_DTYPE_BF16 && in_dtype != KDA_DTYPE_F32) return 0;
    return host_layout(N, T, H, dk, dv, in_dtype, pieces).total;
}

int kda_chunk_fwd_host(const void *q, const void *k, const void *v, const float *g, const float *beta,
                       const int32_t *cu_seqlens, int N, int T, int H, int dk, int dv, const float *initial_state,
                       float *final_state, void *o, float scale, float g_min, int in_dtype, int pieces,
                       void *workspace, size_t workspace_bytes, uint32_t *status, void *stream) {
    if (N < 1 || T < 0 || H < 1 || !cu_seqlens) return KDA_ERR_INVALID_ARG;
    if (!dim_ok(dk) || !dim_ok(dv)) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (in_dtype != KDA_DTYPE_BF16 && in_dtype != KDA_DTYPE_F32) return KDA_ERR_INVALID_ARG;
    if (T > 0 && (!q || !k || !v || !g || !beta || !o)) return KDA_ERR_INVALID_ARG;
    if (cu_seqlens[0] != 0 || cu_seqlens[N] != T) return KDA_ERR_INVALID_ARG;
    for (int n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return KDA_ERR_INVALID_ARG;
    if (pieces < 1) pieces = 4;
    const HostLayout L = host_layout(N, T, H, dk, dv, in_dtype, pieces);
    if (!workspace || workspace_bytes < L.total || !aligned16(workspace)) return KDA_ERR_WORKSPACE;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t es = in_dtype == KDA_DTYPE_BF16 ? 2 : 4;
    const size_t rq = (size_t)H * dk * es, rv = (size_t)H * dv * es, rg = (size_t)H * dk * 4, rb = (size_t)H * 4;
    const size_t sbytes = (size_t)N * H * dk * dv * 4;
    void *dq = ws + L.off_q, *dk_ = ws + L.off_k, *dv_ = ws + L.off_v, *dout = ws + L.off_o;
    float *dg = reinterpret_cast<float *>(ws + L.off_g), *db = reinterpret_cast<float *>(ws + L.off_b);
    int32_t *dcu = reinterpret_cast<int32_t *>(ws + L.off_cu);
    float *ds0 = initial_state ? reinterpret_cast<float *>(ws + L.off_s0) : nullptr;
    float *dsf = final_state ? reinterpret_cast<float *>(ws + L.off_sf) : nullptr;
    auto rows_in = [&](cudaStream_t s, int lo, int hi) -> cudaError_t {
        if (hi <= lo) return cudaSuccess;
        const size_t n = (size_t)(hi - lo);
        cudaError_t e = cudaMemcpyAsync(static_cast<unsigned char *>(dq) + lo * rq,
                                        static_cast<const unsigned char *>(q) + lo * rq, n * rq,
                                        cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(static_cast<unsigned char *>(dk_) + lo * rq,
                                static_cast<const unsigned char *>(k) + lo * rq, n * rq, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(static_cast<unsigned char *>(dv_) + lo * rv,
                                static_cast<const unsigned char *>(v) + lo * rv, n * rv, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(reinterpret_cast<unsigned char *>(dg) + lo * rg,
                                reinterpret_cast<const unsigned char *>(g) + lo * rg, n * rg, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(reinterpret_cast<unsigned char *>(db) + lo * rb,
                                reinterpret_cast<const unsigned char *>(beta) + lo * rb, n * rb,
                                cudaMemcpyHostToDevice, s);
        return e;
    };
    auto rows_out = [&](cudaStream_t s, int lo, int hi) -> cudaError_t {
        if (hi <= lo) return cudaSuccess;
        return cudaMemcpyAsync(static_cast<unsigned char *>(o) + lo * rv,
                               static_cast<const unsigned char *>(dout) + lo * rv, (size_t)(hi - lo) * rv,
                               cudaMemcpyDeviceToHost, s);
    };

    cudaError_t e = cudaSuccess;
    if (!L.pipelined) {  // copy in, the device call, copy out (all on the caller's stream)
        e = cudaMemcpyAsync(dcu, cu_seqlens, (size_t)(N + 1) * 4, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess && ds0) e = cudaMemcpyAsync(ds0, initial_state, sbytes, cudaMemcpyHostToDevice, st);
        if (e == cudaSuccess) e = rows_in(st, 0, T);
        if (e != cudaSuccess) return KDA_ERR_CUDA;
        const int rc = chunk_fwd_impl(dq, dk_, dv_, dg, db, dcu, N, T, H, dk, dv, ds0, dsf, dout, scale, g_min,
                                      in_dtype, KDA_CP_OFF, 0, ws + L.off_area, L.total - L.off_area, 0, 0, nullptr,
                                      status, stream);
        if (rc != KDA_OK) return rc;
        e = rows_out(st, 0, T);
        if (e == cudaSuccess && dsf) e = cudaMemcpyAsync(final_state, dsf, sbytes, cudaMemcpyDeviceToHost, st);
        return cuda_status(e);
    }

    // pieces of slots and the token range each covers (chunks of unit u are
    // slots floor(t0/64) + u + j, in token order)
    const SplitLayout &S = L.S;
    const int P = (S.nslots + S.piece - 1) / S.piece;
    std::vector<int> lo(P, T), hi(P, 0);
    for (int u = 0; u < N; ++u) {
        const int t0 = cu_seqlens[u], t1 = cu_seqlens[u + 1], base = t0 / kChunk + u;
        for (int c = t0; c < t1; c += kChunk) {
            const int pc = (base + (c - t0) / kChunk) / S.piece;
            lo[pc] = lo[pc] < c ? lo[pc] : c;
            const int ce = c + kChunk < t1 ? c + kChunk : t1;
            hi[pc] = hi[pc] > ce ? hi[pc] : ce;
        }
    }
    CopyStreams cs;
    int rc = copy_streams(&cs);
    if (rc != KDA_OK) return rc;
    std::vector<cudaEvent_t> ev(2 * P + 2, nullptr);
    for (auto &x : ev)
        if (cudaEventCreateWithFlags(&x, cudaEventDisableTiming) != cudaSuccess) {
            for (auto &y : ev)
                if (y) cudaEventDestroy(y);
            return KDA_ERR_CUDA;
        }
    cudaEvent_t ev_start = ev[2 * P], ev_done = ev[2 * P + 1];
    kda::ChunkArgs a = {};
    a.q = dq; a.k = dk_; a.v = dv_; a.g = dg; a.beta = db; a.o = dout;
    a.T = T; a.H = H; a.dk = dk; a.dv = dv; a.scale = scale; a.g_min = g_min;
    a.status = status; a.mode = kda::MODE_SEQ; a.cu_seqlens = dcu; a.S_init = ds0; a.S_final = dsf;
    unsigned char *area = ws + L.off_area;
    int2 *list = reinterpret_cast<int2 *>(area + S.off_list);
    int *claim = reinterpret_cast<int *>(area + S.off_claim);
    float *carry = reinterpret_cast<float *>(area + S.off_carry);
    unsigned char *blob = area + S.off_blob;
    // the copy streams start after earlier work on the caller's stream
    e = cudaEventRecord(ev_start, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs.in, ev_start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(cs.out, ev_start, 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dcu, cu_seqlens, (size_t)(N + 1) * 4, cudaMemcpyHostToDevice, cs.in);
    if (e == cudaSuccess && ds0) e = cudaMemcpyAsync(ds0, initial_state, sbytes, cudaMemcpyHostToDevice, cs.in);
    for (int pc = 0; e == cudaSuccess && pc < P; ++pc) {
        e = rows_in(cs.in, lo[pc], hi[pc]);
        if (e == cudaSuccess) e = cudaEventRecord(ev[pc], cs.in);
    }
    for (int pc = 0; e == cudaSuccess && pc < P; ++pc) {
        const int s0 = pc * S.piece, s1 = s0 + S.piece < S.nslots ? s0 + S.piece : S.nslots;
        e = cudaStreamWaitEvent(st, ev[pc], 0);
        if (e == cudaSuccess && pc == 0) e = cudaMemsetAsync(claim, 0, (size_t)P * sizeof(int), st);
        if (e == cudaSuccess && pc == 0)
            e = timed_launch(KDA_KERNEL_CHUNK_LIST, st, [&] { return kda::launch_chunk_list(a, N, S.nslots, list, st); });
        if (e == cudaSuccess)
            e = timed_launch(KDA_KERNEL_CHUNK_PREP, st,
                             [&] { return kda::launch_chunk_prep(a, list, s0, s1, blob, true, claim + pc, false, st); });
        if (e == cudaSuccess)
            e = timed_launch(KDA_KERNEL_CHUNK_WALK, st, [&] {
                return kda::launch_chunk_walk(a, N, blob, s0, s1, carry + (size_t)(pc & 1) * S.carry_stride,
                                              carry + (size_t)((pc + 1) & 1) * S.carry_stride, st);
            });
        if (e == cudaSuccess) e = cudaEventRecord(ev[P + pc], st);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(cs.out, ev[P + pc], 0);
        if (e == cudaSuccess) e = rows_out(cs.out, lo[pc], hi[pc]);
    }
    if (e == cudaSuccess && dsf) e = cudaMemcpyAsync(final_state, dsf, sbytes, cudaMemcpyDeviceToHost, cs.out);
    if (e == cudaSuccess) e = cudaEventRecord(ev_done, cs.out);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev_done, 0);
    for (auto &x : ev) cudaEventDestroy(x);  // released once the work they mark completes
    return cuda_status(e);
}

int kda_kernel_timing_start(void) {
    std::lock_guard<std::mutex> lk(g_timing_mu);
    drop_timed();
    g_timing.store(true);
    return KDA_OK;
}

int kda_kernel_timing_stop(int *launches, float *total_ms, int nkinds) {
    if (nkinds < 0 || (nkinds > 0 && (!launches || !total_ms))) return KDA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_timing_mu);
    g_timing.store(false);
    for (int i = 0; i < nkinds; ++i) {
        launches[i] = 0;
        total_ms[i] = 0.f;
    }
    int rc = KDA_OK;
    for (const TimedLaunch &t : g_timed) {
        float ms = 0.f;
        if (cudaEventSynchronize(t.b) != cudaSuccess || cudaEventElapsedTime(&ms, t.a, t.b) != cudaSuccess) {
            rc = KDA_ERR_CUDA;
            continue;
        }
        if (t.kind >= 0 && t.kind < nkinds) {
            launches[t.kind] += 1;
            total_ms[t.kind] += ms;
        }
    }
    drop_timed();
    return rc;
}

}  // extern "C"
