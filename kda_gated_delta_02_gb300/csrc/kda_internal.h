// kda_internal.h -- launch interfaces between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kda {

enum ChunkMode : int {
    MODE_SEQ = 0,         // one unit per (sequence, head, dv tile)
    MODE_TRANSITION = 1,  // one unit per (segment, head, tile of [M | N])
    MODE_REPLAY = 2,      // one unit per (segment, head, dv tile), seeded from S_in
};

struct ChunkArgs {
    const void *q, *k, *v;
    const float *g, *beta;
    void *o;                    // [T][H][dv] (SEQ / REPLAY)
    int T, H, dk, dv;
    float scale, g_min;
    int mode;
    const int32_t *cu_seqlens;  // SEQ: [N+1]
    const int32_t *seg_table;   // TRANSITION / REPLAY: [P_max][4]
    const int32_t *seg_count;   // device scalar
    int seg_len;                // fixed segment length when seg_table is null
    const float *S_init;        // SEQ: initial_state [N][H][dk][dv] or null
    const float *S_in;          // REPLAY: [P][H][dk][dv]
    float *S_final;             // SEQ / REPLAY: final_state [N][H][dk][dv] or null
    float *M_out, *N_out;       // TRANSITION: [P][H][dk][dk], [P][H][dk][dv]
    uint32_t *status;
    // SEQ / REPLAY: the state every ckpt_every tokens of a sequence (positions
    // ckpt_every * (k + 1), k < ckpt_count) into ckpt [N][ckpt_count][H][dk][dv];
    // null for none.  REPLAY reads the sequence starts from cu_seqlens.
    float *ckpt;
    int ckpt_every, ckpt_count;
};

cudaError_t launch_chunk(const ChunkArgs &a, int units, int dvt, bool in_bf16, cudaStream_t st);

// tcgen05 / tensor-memory version of the chunk kernel (dk = dv = 128, bf16).
bool chunk_tc_supported(const ChunkArgs &a, bool in_bf16);
cudaError_t launch_chunk_tc(const ChunkArgs &a, int units, cudaStream_t st);
// The same prefill as two kernels (chunk_split_tc.cu): the chunk-local
// products of every (chunk, head) in parallel, written as one operand blob of
// kChunkBlobBytes per (chunk, head), then the state walk over the blobs.
// Chunk j of unit u (tokens [t0, t1)) is slot floor(t0 / 64) + u + j.
constexpr unsigned kChunkBlobBytes = 66048;
// Byte offsets inside a blob; every tile 1024-aligned, bf16 tiles in the
// 128-byte swizzled layouts of the tensor-core operands.
constexpr unsigned kBlobW = 0;        // W = T diag(b) K e^gamma: rows = key channel i (128 B of t each)
constexpr unsigned kBlobTB = 16384;   // T diag(b): rows t (128 B of s each)
constexpr unsigned kBlobQT = 24576;   // Q e^gamma: [i / 64][t][64 i]
constexpr unsigned kBlobKT = 40960;   // K e^{gamma_63 - gamma}: [t / 8][i / 64][t % 8][64 i]
constexpr unsigned kBlobBM = 57344;   // B (lower, diagonal included): rows t (128 B of s each)
constexpr unsigned kBlobGam = 65536;  // e^{gamma_63} per key channel, f32 [128]
// list[slot] = {first token, length} for every chunk of units [0, units), 0 elsewhere
cudaError_t launch_chunk_list(const ChunkArgs &a, int units, int nslots, int2 *list, cudaStream_t st);
// blobs of slots [slot0, slot1) into blob[(slot - slot0) * H + h]; claim is a
// device int that is zero when the launch starts (its item counter).  With
// after_walk the launch is a programmatic dependent of the walk launched just
// before it on `st` (it may start while that walk runs; see run_split).  With
// aux (a backward's forward pass) every item also leaves its fp32 T and M^T in
// aux[(slot - slot0) * H + h] ([2][64][64] f32).
cudaError_t launch_chunk_prep(const ChunkArgs &a, const int2 *list, int slot0, int slot1, unsigned char *blob,
                              bool need_q, int *claim, bool after_walk, cudaStream_t st, float *aux = nullptr);
// the chunks of every unit that fall in slots [slot0, slot1); a unit cut at
// slot0 starts from carry_in, one cut at slot1 leaves its state in carry_out
// ([tiles][H][128][128] fp32 each)
// With save_s / save_u (the forward pass a backward uses; o may be null) the
// walk also stores, per (slot, head), its bf16 operand tiles S^T at the chunk
// start (32 KB) and U^T (16 KB), indexed by absolute slot (sequence mode).
cudaError_t launch_chunk_walk(const ChunkArgs &a, int units, const unsigned char *blob, int slot0, int slot1,
                              const float *carry_in, float *carry_out, cudaStream_t st,
                              unsigned char *save_s = nullptr, unsigned char *save_u = nullptr);
// The driver's tensor-map encoder (cuTensorMapEncodeTiled), reached through
// the runtime's entry-point query; null when the driver does not provide it.
void *tensor_map_encoder();

cudaError_t launch_segment_table(const int32_t *cu_seqlens, int N, int T, int seg_len, int P_max,
                                 int32_t *table, int32_t *seq_first, int32_t *seg_count,
                                 uint32_t *status, cudaStream_t st);

// Ordered composition over chains.  Chain c covers segments
// [first[c], first[c+1]) when `first` is given, else [c*P, (c+1)*P); per head.
struct ComposeArgs {
    const float *M, *Nm;
    const float *S0;      // [chains][H][dk][dv] or null
    float *S_in;          // [P_total][H][dk][dv] or null
    float *S_final;       // [chains][H][dk][dv] or null
    const int32_t *first; // [chains+1] device or null
    int P;                // segments per chain when first == null
    int chains, H, dk, dv;
};
cudaError_t launch_compose(const ComposeArgs &a, cudaStream_t st);

// Backward of the prefill (chunk_bwd.cu), dk = dv = d in {64, 128}.
struct BwdArgs {
    const void *q, *k, *v, *dout;  // [T][H][d], bf16 or f32
    const float *g, *beta;         // [T][H][d], [T][H]
    const int32_t *cu_seqlens;     // [N+1]
    const float *S0, *dS_final;    // [N][H][d][d] or null (zero)
    float *dq, *dk, *dv, *dg, *dbeta, *dS0;  // dS0 may be null
    float *ckpt;                   // [floor(T/64) + N slots][H][d][d] chunk-start states
    float *scratch;                // [min(N H, kBwdMaxCtas)][64][d][d] states of the chunk being differentiated
    float *partials;               // [min(N H, kBwdMaxCtas) d/32][2][chunk_bwd_partial_floats(d)] column
                                   // partials of the split form (null: the whole form)
    float *wbuf;                   // [T][H][d] w = v - p of every token (pass 1 -> pass 2)
    int N, T, H;
    float scale, g_min;
    uint32_t *status;
};
// the backward keeps at most this many (sequence, head) units in flight (one
// scratch slot each; a whole-form CTA or a split-form cluster per unit)
constexpr int kBwdMaxCtas = 160;
// floats of one chunk's column partials of one split-form CTA
size_t chunk_bwd_partial_floats(int d);
cudaError_t launch_chunk_bwd(const BwdArgs &a, int d, bool bf16, cudaStream_t st);

// Backward on the tensor cores (chunk_bwd_tc.cu): dk = dv = 128, bf16 q, k,
// v, dout.  The forward pass (chunk-local kernel with aux, walk saving its
// tiles) fills blob, aux, save_s and save_u for every slot; the reverse walk
// fills save_ds and save_du and writes dS0; the chunk kernel writes dq, dk,
// dv, dg, dbeta.  Per (slot, head): blob kChunkBlobBytes, aux 32 KB, save_s
// and save_ds 32 KB, save_u and save_du 16 KB.
struct BwdTcArgs {
    const void *q, *k, *v, *dout;
    const float *g, *beta;
    const int32_t *cu_seqlens;
    int N, T, H;
    float scale, g_min;
    const float *dS_final;
    float *dq, *dk, *dv, *dg, *dbeta, *dS0;
    const int2 *list;
    const unsigned char *blob;
    const float *aux;
    unsigned char *save_s, *save_u, *save_ds, *save_du;
    uint32_t *status;
};
// The reverse walk over the chunks in slots [slot0, slot1), newest first; a
// sequence cut at slot1 starts from carry_in, one cut at slot0 leaves its
// state gradient in carry_out ([H][128][128] f32 each).
// Context-parallel segments for the reverse walk (one piece): the segment
// table of the forward's schedule; the first pass starts every segment from
// zero (dS_in null) and leaves r_out, the second starts from dS_in and keeps
// the tiles (save).
struct BwdSegments {
    const int32_t *table, *count;
    int P_max;
    const float *dS_in;
    float *r_out;
    bool save;
};
cudaError_t launch_bwd_walk(const BwdTcArgs &a, int slot0, int slot1, const float *carry_in, float *carry_out,
                            cudaStream_t st, const BwdSegments *sg = nullptr);
// dS' over a sequence's segments, last to first: dS'_start = M_p^T dS'_end + r_p
// (M [P][H][dk][dk] the forward transitions, first [N+1] each sequence's
// first segment); dS_end [P][H][dk][dv] raw dS' at each segment end, dS0 =
// scale dS' at the sequence start (or null).
cudaError_t launch_bwd_compose(const float *M, const float *r, const int32_t *first, const int32_t *cu,
                               const float *dS_final, float *dS_end, float *dS0, int N, int H, float scale,
                               cudaStream_t st);
// The chunk gradients of slots [slot0, slot1); claim is a device int that is
// zero when the launch starts.  With after_walk the launch is a programmatic
// dependent of the reverse walk launched just before it on `st` (it may start
// while that walk runs: it reads only what earlier launches wrote).
cudaError_t launch_bwd_chunk(const BwdTcArgs &a, int slot0, int slot1, int *claim, bool after_walk,
                             cudaStream_t st);

struct VerifyArgs {
    void *state, *tail;
    const float *conv_w;
    const void *cached_qkv, *cached_g, *cached_b;
    const int32_t *accepted;
    const int32_t *draft_len;  // [R] drafts per request, or null (every request has Wd)
    const void *new_qkv, *new_g, *new_b;
    const float *out_w;
    void *o;
    int R, H, dk, dv, W, Wd;
    float scale, g_min, eps_in, eps_out;
    int conv_act;
    uint32_t *status;
};
cudaError_t launch_verify(const VerifyArgs &a, cudaStream_t st);
// tcgen05 / tensor-memory version of the verify kernel (dk = dv = 128).
cudaError_t launch_verify_tc(const VerifyArgs &a, cudaStream_t st);
// Single-token decode (Wd = 0) on the CUDA cores (dk = dv = 64 or 128).
cudaError_t launch_decode_token(const VerifyArgs &a, cudaStream_t st);

}  // namespace kda
