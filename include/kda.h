/*
 * kda.h -- C ABI of the KDA (gated delta rule) hot path for NVIDIA GB300 (sm_103a).
 *
 * The recurrence, per head, with a fixed-size state S in R^{dk x dv}
 * ("Noyaux KDA et FlashKDA", section "Le conflit fondamental"):
 *     S_t = (I - b_t k_t k_t^T) Diag(exp g_t) S_{t-1} + b_t k_t v_t^T,
 *     o_t = scale * S_t^T q_t,
 * where g_t in R^{dk} is a per-channel log-decay acting on the key axis and
 * floored at g_min = -5 per token and channel ("Noyaux KDA et FlashKDA",
 * section "Le role de la decroissance bornee").
 *
 * Conventions shared by every call:
 *  - Ownership: the caller allocates and owns all memory.  Pointers named
 *    "device" must be device memory of the current CUDA device; the library
 *    never allocates device memory, except inside caller-provided workspace.
 *  - Layouts: contiguous, row-major, token-major ("THD"):
 *        q, k, g [T][H][dk], v, o [T][H][dv], beta [T][H];
 *    states head-contiguous [.., H, dk, dv] with dv fastest ("Inference :
 *    cache KV, decodage, quantification": each head's state is one
 *    self-contained byte stream).
 *  - Alignment: every tensor pointer must be 16-byte aligned.
 *  - Streams: every call takes a cudaStream_t passed as void* (NULL = the
 *    legacy default stream), enqueues its kernels there and returns without
 *    synchronising.
 *  - Errors: every call returns an int status.  Host-side validation runs
 *    before any launch: on failure nothing is enqueued.  KDA_ERR_CUDA means a
 *    launch failed (cudaGetLastError).  Conditions only visible on the device
 *    (bad cu_seqlens, out-of-range accepted lengths) set bits in the optional
 *    device status word `status` (a uint32 the caller zeroes and reads back
 *    when convenient); the affected work unit is skipped.  No kernel traps.
 *  - Supported shapes: dk, dv in {64, 128}; H >= 1.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KDA_OK 0
#define KDA_ERR_INVALID_ARG (-1)
#define KDA_ERR_UNSUPPORTED_SHAPE (-2)
#define KDA_ERR_ALIGNMENT (-3)
#define KDA_ERR_WORKSPACE (-4)
#define KDA_ERR_CUDA (-5)
#define KDA_ERR_SCRATCH_LIMIT (-6)

#define KDA_DTYPE_BF16 0
#define KDA_DTYPE_F32 1

#define KDA_CONV_NONE 0
#define KDA_CONV_SILU 1

#define KDA_CP_OFF 0
#define KDA_CP_ON 1
#define KDA_CP_AUTO (-1)

/* Bits of the device status word. */
#define KDA_STATUS_BAD_SEQLENS 0x1u      /* cu_seqlens not monotone / out of [0, T] */
#define KDA_STATUS_BAD_ACCEPTED_LEN 0x2u /* accepted_len[r] outside [0, Wd]        */
#define KDA_STATUS_SEGMENT_OVERFLOW 0x4u /* segment table larger than planned      */
#define KDA_STATUS_TIMEOUT 0x8u          /* a bounded on-chip wait gave up; unit left unfinished */
#define KDA_STATUS_BAD_DRAFT_LEN 0x10u   /* draft_len[r] outside [0, Wd]                         */

/* Kernel families, for kda_kernel_timing_stop. */
#define KDA_KERNEL_CHUNK_LIST 0      /* chunk slot list of the two-kernel prefill */
#define KDA_KERNEL_CHUNK_PREP 1      /* chunk-local products of the two-kernel prefill */
#define KDA_KERNEL_CHUNK_WALK 2      /* state walk of the two-kernel prefill */
#define KDA_KERNEL_CHUNK_TC 3        /* one-kernel tcgen05 prefill */
#define KDA_KERNEL_CHUNK_MMA 4       /* warp-MMA prefill (d = 64, f32 inputs) */
#define KDA_KERNEL_SEGMENT_COMPOSE 5 /* CP composition */
#define KDA_KERNEL_SEGMENT_TABLE 6   /* CP segment table */
#define KDA_KERNEL_VERIFY 7          /* kda_decode_verify_replay (verify or single-token decode) */
#define KDA_KERNEL_CHUNK_BWD 8       /* kda_chunk_bwd on the CUDA cores (d = 64 or f32 inputs) */
#define KDA_KERNEL_BWD_WALK 9        /* kda_chunk_bwd, tensor cores: reverse state walk */
#define KDA_KERNEL_BWD_CHUNK 10      /* kda_chunk_bwd, tensor cores: chunk gradients */
#define KDA_KERNEL_BWD_COMPOSE 11    /* kda_chunk_bwd_cp: state gradient over the segments */
#define KDA_KERNEL_KINDS 12

/* Human-readable name of a return status. Never NULL. */
const char *kda_status_string(int status);

/* ABI version (major*100 + minor). */
int kda_version(void);

/*
 * Chunkwise prefill / training forward ("Noyaux KDA et FlashKDA", section
 * "FlashKDA : le noyau par blocs": parallel inside a 64-token chunk, serial
 * between chunks; the floor makes every causal tile a dense product, section
 * "Le role de la decroissance bornee").
 *
 *  q, k, v      device, [T][H][dk] / [T][H][dv], dtype in_dtype (bf16 | f32).
 *  g            device, f32 [T][H][dk], raw log-decay; floored at g_min on load
 *               (a NaN takes the floor, as an IEEE maximum does).
 *  beta         device, f32 [T][H].
 *  cu_seqlens   device, int32 [N+1], N sequences packed along T
 *               (cu_seqlens[0] = 0, non-decreasing, cu_seqlens[N] = T).
 *               Chunks restart at every sequence start.
 *  initial_state device f32 [N][H][dk][dv] or NULL (zero state).
 *  final_state  device f32 [N][H][dk][dv] or NULL (not written).
 *  o            device, [T][H][dv], dtype in_dtype.
 *  scale        multiplies o (1.0 for the plain rule).
 *  g_min        decay floor (-5).
 *  cp_mode      KDA_CP_OFF: one pass per (sequence, head).
 *               KDA_CP_ON: intra-device context parallelism ("Noyaux KDA et
 *               FlashKDA", section "Le parallelisme de contexte
 *               intra-appareil"): segments of segment_len tokens are turned
 *               into independent affine transitions (M, N), composed in order
 *               per (sequence, head), then replayed in parallel from their
 *               exact initial states (4 launches).
 *               KDA_CP_AUTO: CP when (sequence, head) units are too few to
 *               fill the GPU and sequences are long.
 *  segment_len  CP segment length in tokens (multiple of 64), or 0 = automatic:
 *               segments of at least 1,024 tokens, about one (segment, head)
 *               unit per SM at dk = dv = 128 (the state walk holds one block
 *               per SM), two per SM otherwise.
 *  workspace    device scratch of at least kda_chunk_fwd_workspace_size(...)
 *               bytes (may be NULL when that size is 0).  Contents on entry
 *               are ignored; on exit they are unspecified.  With bf16 inputs
 *               and dk = dv = 128, a workspace of at least
 *               kda_chunk_fwd_prep_workspace_size(...) bytes (or any size
 *               with room for one slot, run in pieces) selects the
 *               two-kernel form: the chunk-local products of every (chunk,
 *               head) (decays, causal tiles, the dependency inverse, W, the
 *               decayed q and k) run first, in parallel over all chunks, into
 *               an operand area of the workspace; then each (sequence or
 *               segment, head) walks its chunks with only the state products
 *               left on its serial path.  Same results as the one-kernel form
 *               (same operations in the same order); a smaller workspace runs
 *               the one-kernel form.
 *  status       device uint32 status word or NULL.
 */
int kda_chunk_fwd(const void *q, const void *k, const void *v, const float *g,
                  const float *beta, const int32_t *cu_seqlens, int N, int T, int H, int dk,
                  int dv, const float *initial_state, float *final_state, void *o, float scale,
                  float g_min, int in_dtype, int cp_mode, int segment_len, void *workspace,
                  size_t workspace_bytes, uint32_t *status, void *stream);

/*
 * kda_chunk_fwd that also emits intermediate states: prefix-cache resume
 * points ("Dentro de los esfuerzos de optimizacion de Kimi K3", section 5:
 * states kept at block-aligned positions so that a later request sharing the
 * prefix continues from them).  Same arguments and results as kda_chunk_fwd,
 * plus:
 *  ckpt_every  positive multiple of 64: a checkpoint is the state after token
 *              ckpt_every * (k + 1) of a sequence (positions counted from the
 *              sequence start), k = 0 .. ckpt_count - 1.
 *  ckpt_count  checkpoints kept per sequence; positions past a sequence's end
 *              are not written (those slots keep their contents).
 *  ckpt        device f32 [N][ckpt_count][H][dk][dv], or NULL when ckpt_count = 0.
 * Works with context parallelism on or off (the replay pass writes them).
 * Invalid ckpt arguments return KDA_ERR_INVALID_ARG before any launch.
 */
int kda_chunk_fwd_ckpt(const void *q, const void *k, const void *v, const float *g,
                       const float *beta, const int32_t *cu_seqlens, int N, int T, int H,
                       int dk, int dv, const float *initial_state, float *final_state, void *o,
                       float scale, float g_min, int in_dtype, int cp_mode, int segment_len,
                       void *workspace, size_t workspace_bytes, int ckpt_every, int ckpt_count,
                       float *ckpt, uint32_t *status, void *stream);

/* Workspace bytes kda_chunk_fwd needs for these arguments (0 when cp_mode
 * resolves to OFF).  Pure host arithmetic. */
size_t kda_chunk_fwd_workspace_size(int N, int T, int H, int dk, int dv, int cp_mode,
                                    int segment_len);

/* Workspace bytes that select kda_chunk_fwd's two-kernel form (bf16 inputs,
 * dk = dv = 128) in the layout the call prefers: the CP scratch above, then a
 * slot list (8 bytes per 64-token chunk slot; floor(T / 64) + units slots,
 * units = sequences or segments), one 4-byte item counter per slot, two carry
 * states (2 x 2 x H x 128 x 128 f32) and the operand blobs (66,048 bytes per
 * slot and head).  A call whose walks leave SMs idle (units x H below the SM
 * count) with at least 64 slots asks for two blob buffers of a quarter of the
 * slots each: its four pieces are pipelined, the chunk-local kernel of piece
 * p + 1 running as a programmatic dependent launch beside the walk of piece
 * p.  Other calls, and context-parallel ones (whose transition blobs then
 * serve the replay), ask for all slots in one piece.  Blobs are capped at 16
 * GiB.  kda_chunk_fwd uses whatever workspace it is given: room for fewer
 * slots runs smaller pieces (pipelined while two slots fit, else one at a
 * time); room for none runs the one-kernel form.  Equals
 * kda_chunk_fwd_workspace_size for other shapes.  Pure host arithmetic (it
 * reads the SM count of the current device); this form has no counterpart
 * on the pages beyond the chunk algebra it reorders and overlaps. */
size_t kda_chunk_fwd_prep_workspace_size(int N, int T, int H, int dk, int dv, int cp_mode,
                                         int segment_len);

/* The segment length (tokens) and CP decision kda_chunk_fwd would use:
 * returns 0 when CP is off, else the segment length. Pure host arithmetic. */
int kda_chunk_fwd_plan(int N, int T, int H, int dk, int dv, int cp_mode, int segment_len);

/*
 * kda_chunk_fwd (cp off) on host buffers, with the transfers overlapped with
 * the kernels: q, k, v, g, beta, cu_seqlens, initial_state, final_state and o
 * are HOST pointers (page-locked for the copies to run asynchronously) with
 * kda_chunk_fwd's layouts; workspace is device memory of at least
 * kda_chunk_fwd_host_workspace_size(...) bytes (device copies of inputs and
 * outputs and the two-kernel area).  With bf16 inputs and dk = dv = 128 the
 * chunk slots run in `pieces` equal pieces (0: 4): while piece p's chunk-local
 * kernel and walk run on `stream`, piece p+1's input rows are copied in and
 * piece p-1's output rows copied out, on two internal streams of the library
 * ordered by events; other shapes copy in, run kda_chunk_fwd and copy out on
 * `stream`.  When `stream` completes, o and final_state hold the results.
 * cu_seqlens must satisfy cu_seqlens[0] = 0, non-decreasing, cu_seqlens[N] =
 * T (checked on the host: KDA_ERR_INVALID_ARG).  A workspace smaller than the
 * size returns KDA_ERR_WORKSPACE.  Results are those of kda_chunk_fwd with
 * the same pieces (bit for bit).  The pages have no counterpart: this is an
 * interface for callers whose inputs live in host memory.
 */
int kda_chunk_fwd_host(const void *q, const void *k, const void *v, const float *g,
                       const float *beta, const int32_t *cu_seqlens, int N, int T, int H,
                       int dk, int dv, const float *initial_state, float *final_state, void *o,
                       float scale, float g_min, int in_dtype, int pieces, void *workspace,
                       size_t workspace_bytes, uint32_t *status, void *stream);
size_t kda_chunk_fwd_host_workspace_size(int N, int T, int H, int dk, int dv, int in_dtype,
                                         int pieces);

/*
 * Backward of kda_chunk_fwd (training; "Noyaux KDA et FlashKDA", section
 * "FlashKDA : le noyau par blocs" names it as the chunk kernel's other use):
 * the gradients of a loss L with respect to every input, given dL/do and
 * dL/dS_final.  Two forms, chosen by shape and input type:
 *
 * bf16 inputs at d = 128: the chunk (WY) form on the tensor cores.  For a
 * 64-token chunk entered with state S (gamma the running sum of the floored
 * log-decays, K~ = K e^gamma, Q~ = Q e^gamma, K^ = K e^{gamma_63 - gamma},
 * M = strict_lower(K~ (K e^-gamma)^T), T = (I + diag(b) M)^{-1}, TB = T diag(b),
 * W = TB K~, B = lower(Q~ (K e^-gamma)^T)):
 *     Vres = V - K~ S,  U = TB Vres,  O = scale (Q~ S + B U),  S_C = Diag(e^{gamma_63}) S + K^^T U.
 * A forward pass (the two-kernel prefill's kernels, in pipelined pieces)
 * keeps every chunk's operand blob, its fp32 T and M, and the bf16 state and
 * U tiles; a reverse walk per (sequence, head) carries dS (arriving at each
 * chunk end) backwards, dU = scale B^T dO + K^ dS_C and
 * dS = scale Q~^T dO + Diag(e^{gamma_63}) dS_C - W^T dU, on the same blobs;
 * then every chunk's token gradients are formed in parallel (the reverse of
 * each forward step: dVres = TB^T dU = dv, dTB = dU Vres^T,
 * dA = strict_lower(-T^T dTB diag(b) T^T), dB = scale lower(dO U^T), the causal
 * tiles' gradients through the forward's 16-token block anchoring, and the
 * reverse cumulative sum of the log-decay gradient).  Products take bf16
 * operands with fp32 accumulation (T diag(b) keeps a second bf16 part);
 * gradients are within 1e-2 of the fp64 reverse mode, normwise per head.
 *
 * d = 64, or fp32 inputs: the reverse mode of the token recurrence in fp32 on
 * the CUDA cores (S before a token, S' after it, D = Diag(e^{max(g, g_min)}),
 * X = D S, p = X^T k, u = beta (v - p), S' = X + k u^T, o = scale S'^T q;
 * G = dL/dS'):
 *     G += scale q do^T;  dq = scale S' do;  du = G^T k;  dv = beta du;
 *     dbeta = du . (v - p);  dk = G u - beta X du;  dX = G - beta k du^T;
 *     dg_i = sum_j dX_ij X_ij, 0 where g_i < g_min;  G <- D dX;  dS0 = G at the start,
 * each (sequence, head) walked by a cluster of d/32 CTAs, one per 32 value
 * columns of the state, whose per-column partial sums are added in a fixed
 * order; states are recomputed from chunk-start checkpoints.
 *
 * Both forms are deterministic (the same inputs give the same bits).
 *  q, k, v, g, beta, cu_seqlens, N, T, H, initial_state, scale, g_min,
 *  in_dtype   as kda_chunk_fwd (dk = dv = 64 or 128; cp off).
 *  dout       device [T][H][dv], in_dtype: dL/do.
 *  dS_final   device f32 [N][H][dk][dv] or NULL (zero): dL/dS_final.
 *  dq, dk, dv device f32 [T][H][d]; dg device f32 [T][H][dk] (w.r.t. the raw
 *             g: zero where g < g_min; a NaN g gets the gradient of g = g_min);
 *             dbeta device f32 [T][H]; dS0 device f32 [N][H][dk][dv] or NULL.
 *  workspace  device scratch of at least kda_chunk_bwd_workspace_size(...)
 *             bytes, 256-byte aligned parts.  Tensor-core form, with
 *             S = floor(T/64) + N chunk slots: the slot list (S x 8 B),
 *             item counters (256 B), two carry states per head
 *             (2 x H x 128 x 128 f32), then per (slot, head) the operand
 *             blob (66,048 B), T and M^T (f32, 32 KB), the bf16 tiles of
 *             the state and U (32 + 16 KB) and of the state gradient and dU
 *             (32 + 16 KB).  CUDA-core form: S x H chunk checkpoints and
 *             min(N x H, 160) x 64 states, d x d f32 each, then
 *             min(N x H, 160) x d/32 x 2 buffers of 64 x (3d + 1) f32 column
 *             partials, then T x H x d f32 (w = v - p of every token).  The
 *             size is the larger of the two at d = 128 (independent of
 *             in_dtype); KDA_ERR_WORKSPACE when smaller.
 * Invalid cu_seqlens set KDA_STATUS_BAD_SEQLENS; that sequence is skipped.
 */
int kda_chunk_bwd(const void *q, const void *k, const void *v, const float *g, const float *beta,
                  const int32_t *cu_seqlens, int N, int T, int H, int dk, int dv,
                  const float *initial_state, const void *dout, const float *dS_final, float *dq,
                  float *dk_, float *dv_, float *dg, float *dbeta, float *dS0, float scale,
                  float g_min, int in_dtype, void *workspace, size_t workspace_bytes,
                  uint32_t *status, void *stream);
size_t kda_chunk_bwd_workspace_size(int N, int T, int H, int dk, int dv);

/*
 * kda_chunk_bwd with the prefill's context-parallel schedule for long
 * sequences ("Noyaux KDA et FlashKDA", section "Le parallelisme de contexte
 * intra-appareil", in reverse): cp_mode and segment_len as kda_chunk_fwd.
 * When the call is cut into segments (bf16, d = 128), the forward pass runs
 * as the CP prefill does (every segment's transition S_end = M S_start + N,
 * the ordered composition, the replay keeping its tiles); the state gradient
 * is affine over a segment too, dS_start = M^T dS_end + r with r the
 * gradient a segment reaches from zero at its end, so every segment's r is
 * walked in parallel, a short scan composes them last to first per
 * (sequence, head), and every segment is walked again from its exact end
 * gradient; then the chunk gradients as in kda_chunk_bwd.  Otherwise (CP off
 * or declined, other shapes) it is kda_chunk_bwd.  Results agree with
 * kda_chunk_bwd within the tensor-core form's rounding (1e-2 of the fp64
 * reverse mode).
 *  cp_mode    KDA_CP_AUTO cuts the call when kda_chunk_fwd's automatic mode
 *             would, and segment_len 0 picks kda_chunk_fwd's length (about
 *             one (segment, head) unit per SM).
 *  workspace  at least kda_chunk_bwd_cp_workspace_size(...) bytes: the CP
 *             prefill's area, the tensor-core layout over S = floor(T/64) +
 *             P_max slots, and 2 x P_max x H x 128 x 128 f32 (r and the
 *             segment-end gradients); KDA_ERR_WORKSPACE when smaller.
 */
int kda_chunk_bwd_cp(const void *q, const void *k, const void *v, const float *g,
                     const float *beta, const int32_t *cu_seqlens, int N, int T, int H, int dk,
                     int dv, const float *initial_state, const void *dout, const float *dS_final,
                     float *dq, float *dk_, float *dv_, float *dg, float *dbeta, float *dS0,
                     float scale, float g_min, int in_dtype, int cp_mode, int segment_len,
                     void *workspace, size_t workspace_bytes, uint32_t *status, void *stream);
size_t kda_chunk_bwd_cp_workspace_size(int N, int T, int H, int dk, int dv, int cp_mode,
                                       int segment_len);

/*
 * The training pair of the tensor-core form (dk = dv = 128, bf16 inputs;
 * KDA_ERR_UNSUPPORTED_SHAPE otherwise): the forward pass that kda_chunk_bwd
 * runs first, returning the prefill's outputs as well, then the reverse pass
 * alone.  A training step calls kda_chunk_fwd_train once and
 * kda_chunk_bwd_saved once instead of kda_chunk_fwd and kda_chunk_bwd (which
 * runs the forward pass again).
 *  kda_chunk_fwd_train: arguments and results as kda_chunk_fwd (cp off), and
 *             saved: device buffer of at least
 *             kda_chunk_bwd_workspace_size(N, T, H, 128, 128) bytes that
 *             receives the slot list, every chunk's operand blob, T and M^T,
 *             and the walk's state and U tiles (the tensor-core layout of
 *             kda_chunk_bwd's workspace).  o and final_state are those of
 *             kda_chunk_fwd bit for bit.
 *  kda_chunk_bwd_saved: arguments as kda_chunk_bwd without initial_state
 *             (the state tiles are saved), and saved as written by
 *             kda_chunk_fwd_train with the same q, k, v, g, beta,
 *             cu_seqlens, N, T, H, scale and g_min (the library does not
 *             check that they are the same); it also holds the reverse
 *             pass's own tiles, so it is written.  Results are those of
 *             kda_chunk_bwd on the same inputs bit for bit.
 * KDA_ERR_WORKSPACE when saved is smaller than the size.
 */
int kda_chunk_fwd_train(const void *q, const void *k, const void *v, const float *g,
                        const float *beta, const int32_t *cu_seqlens, int N, int T, int H, int dk,
                        int dv, const float *initial_state, float *final_state, void *o,
                        float scale, float g_min, int in_dtype, void *saved, size_t saved_bytes,
                        uint32_t *status, void *stream);
int kda_chunk_bwd_saved(const void *q, const void *k, const void *v, const float *g,
                        const float *beta, const int32_t *cu_seqlens, int N, int T, int H, int dk,
                        int dv, const void *dout, const float *dS_final, float *dq, float *dk_,
                        float *dv_, float *dg, float *dbeta, float *dS0, float scale, float g_min,
                        int in_dtype, void *saved, size_t saved_bytes, uint32_t *status,
                        void *stream);

/*
 * The training pair with kda_chunk_bwd_cp's context-parallel schedule: the
 * forward pass kda_chunk_bwd_cp runs first (segment table, operand blobs with
 * T and M^T, transitions, their composition, the replay keeping its tiles),
 * returning the prefill's outputs as well, then its reverse pass alone.
 * Arguments as kda_chunk_fwd_train / kda_chunk_bwd_saved plus cp_mode and
 * segment_len (as kda_chunk_bwd_cp; both calls must get the same values, and
 * the same inputs, which the library does not check).
 *  saved   device buffer of at least kda_chunk_bwd_cp_workspace_size(N, T,
 *          H, 128, 128, cp_mode, segment_len) bytes; kda_chunk_fwd_train_cp
 *          writes it, kda_chunk_bwd_saved_cp reads it and writes its own
 *          parts (segment gradients, state-gradient tiles).
 * When the call is not cut into segments they are kda_chunk_fwd_train and
 * kda_chunk_bwd_saved.  Results are kda_chunk_fwd's (cp_mode, segment_len)
 * outputs and kda_chunk_bwd_cp's gradients bit for bit (same kernels on the
 * same operands).  KDA_ERR_WORKSPACE when saved is smaller than the size.
 */
int kda_chunk_fwd_train_cp(const void *q, const void *k, const void *v, const float *g,
                           const float *beta, const int32_t *cu_seqlens, int N, int T, int H,
                           int dk, int dv, const float *initial_state, float *final_state, void *o,
                           float scale, float g_min, int in_dtype, int cp_mode, int segment_len,
                           void *saved, size_t saved_bytes, uint32_t *status, void *stream);
int kda_chunk_bwd_saved_cp(const void *q, const void *k, const void *v, const float *g,
                           const float *beta, const int32_t *cu_seqlens, int N, int T, int H,
                           int dk, int dv, const void *dout, const float *dS_final, float *dq,
                           float *dk_, float *dv_, float *dg, float *dbeta, float *dS0, float scale,
                           float g_min, int in_dtype, int cp_mode, int segment_len, void *saved,
                           size_t saved_bytes, uint32_t *status, void *stream);

/*
 * Segment transitions of one sequence ("Noyaux KDA et FlashKDA", section "Le
 * parallelisme de contexte intra-appareil": the transition of each segment is
 * evaluated independently of the incoming state).  Exported for tests and
 * debugging; kda_chunk_fwd's CP path runs the same kernel.
 * Tokens [0, T) of one sequence are cut into P = ceil(T / segment_len)
 * segments; per segment p and head h:
 *     M[p][h] = A_last ... A_first   (A_t = (I - b_t k_t k_t^T) Diag(exp g_t)),
 *     Nmat[p][h] = state reached from S = 0 over the segment.
 *  k, v, g, beta  device, as in kda_chunk_fwd (single sequence, length T).
 *  M              device f32 [P][H][dk][dk];  Nmat device f32 [P][H][dk][dv].
 */
int kda_segment_transition(const void *k, const void *v, const float *g, const float *beta,
                           int T, int H, int dk, int dv, int segment_len, float *M, float *Nmat,
                           float g_min, int in_dtype, void *stream);

/*
 * Exact ordered composition of segment transitions, per head ("Dentro de los
 * esfuerzos de optimizacion de Kimi K3", section 5: group summaries are
 * scanned in order to give every group its exact initial state):
 *     S_in[p] = S_{p-1},   S_p = M[p] S_{p-1} + Nmat[p],   S_{-1} = S0 (or 0).
 *  M      device f32 [P][H][dk][dk];  Nmat device f32 [P][H][dk][dv].
 *  S0     device f32 [H][dk][dv] or NULL.
 *  S_in   device f32 [P][H][dk][dv] or NULL (initial state of each segment).
 *  S_final device f32 [H][dk][dv] or NULL.
 * Arithmetic is fp32 with fp32 accumulation.
 */
int kda_segment_compose(const float *M, const float *Nmat, const float *S0, float *S_in,
                        float *S_final, int P, int H, int dk, int dv, void *stream);

/*
 * Fused speculative-decode verify with replay from projected inputs, one KDA
 * layer, R requests ("Noyaux d'inference", section 1 "Le decodage KDA",
 * subsections "La solution : rejouer plutot que sauvegarder" and "La fusion").
 * Per request r the token sequence is: cached rows 0..a-1 (accepted drafts of
 * the previous window, replayed), new row 0 (bonus token), new rows 1..Wd
 * (next draft window), a = accepted_len[r].  For each token, in one kernel:
 * depthwise causal short conv of width W over the pre-conv q|k|v channels
 * (the W-1 previous rows come from conv_tail, then from earlier tokens),
 * optional SiLU, L2 norm of q and k over dk (eps_in), gates
 * g = max(-softplus(g_raw), g_min), b = sigmoid(b_raw), the recurrence, and
 * for the bonus and draft tokens the per-head RMSNorm of o over dv (eps_out)
 * times out_norm_w.  The state reached after the bonus token is written back
 * to `state` (bf16, round to nearest even) and conv_tail receives the W-1
 * most recent pre-conv rows up to and including the bonus row (bitwise
 * copies).  Draft tokens never touch HBM state.
 *
 *  state        device bf16 [R][H][dk][dv], in/out.
 *  conv_tail    device bf16 [R][W-1][Cq], in/out, Cq = H*(2*dk+dv), rows oldest
 *               first; channel order q (H*dk) | k (H*dk) | v (H*dv), head-major.
 *  conv_w       device f32 [Cq][W]; y_t = sum_j conv_w[c][j] x_{t-(W-1)+j}[c].
 *  cached_qkv   device bf16 [R][Wd][Cq];  cached_g bf16 [R][Wd][H*dk];
 *  cached_beta  bf16 [R][Wd][H]  -- the previous window's draft rows.
 *  accepted_len device int32 [R], valid range [0, Wd]; a request outside it
 *               is skipped (state, tail and o untouched) and
 *               KDA_STATUS_BAD_ACCEPTED_LEN is set.
 *  new_qkv      device bf16 [R][Wd+1][Cq];  new_g bf16 [R][Wd+1][H*dk];
 *  new_beta     bf16 [R][Wd+1][H]  -- row 0 bonus, rows 1..Wd drafts.
 *               A NaN raw gate g takes the floor g_min (as an IEEE maximum).
 *  out_norm_w   device f32 [dv].
 *  o            device bf16 [R][Wd+1][H][dv]: rows for bonus + drafts.
 *  Limits: W in [1, 4] and Wd in [0, 7], so that the a + 1 + Wd <= 2*Wd + 1
 *  tokens of a request fit one 16-token tile on chip.
 * The caller swaps the cached and new buffers between steps (new rows 1..Wd
 * become the next cached rows); the kernel copies no projection.
 */
int kda_decode_verify_replay(void *state, void *conv_tail, const float *conv_w,
                             const void *cached_qkv, const void *cached_g,
                             const void *cached_beta, const int32_t *accepted_len,
                             const void *new_qkv, const void *new_g, const void *new_beta,
                             const float *out_norm_w, void *o, int R, int H, int dk, int dv,
                             int W, int Wd, float scale, float g_min, float eps_in,
                             float eps_out, int conv_act, uint32_t *status, void *stream);

/*
 * kda_decode_verify_replay for a ragged batch: request r carries its own
 * number of drafts draft_len[r] in [0, Wd] ("Dentro de los esfuerzos de
 * optimizacion de Kimi K3", section 5: uniform batches take a specialised
 * path, irregular batches keep a dynamic one; the pages' drafts range over
 * 3-7).  Arrays keep their Wd-sized layouts; request r's verify sequence is
 * its a_r replayed rows, the bonus and new rows 1..draft_len[r]; new rows past
 * draft_len[r] are never read into the recurrence (they may hold anything,
 * NaN included) and its o rows past draft_len[r] are not written.  State and
 * conv tail are written back after the bonus, as in the uniform call.
 *  draft_len  device int32 [R]; NULL = every request has Wd drafts (the
 *             uniform call).  A count outside [0, Wd] sets
 *             KDA_STATUS_BAD_DRAFT_LEN and skips the request (state, tail and
 *             o untouched).  With Wd = 0 every count must be 0.
 * Other arguments, layouts and errors as kda_decode_verify_replay.
 */
int kda_decode_verify_replay_ragged(void *state, void *conv_tail, const float *conv_w,
                                    const void *cached_qkv, const void *cached_g,
                                    const void *cached_beta, const int32_t *accepted_len,
                                    const int32_t *draft_len, const void *new_qkv,
                                    const void *new_g, const void *new_beta,
                                    const float *out_norm_w, void *o, int R, int H, int dk,
                                    int dv, int W, int Wd, float scale, float g_min,
                                    float eps_in, float eps_out, int conv_act,
                                    uint32_t *status, void *stream);

/*
 * Context-parallel prefill that allocates nothing.  (The pages have no
 * counterpart: this is an interface for callers of this library.)
 *
 * Some callers cannot call cudaMalloc or hand over a workspace: for example a
 * serving loop whose host forbids device allocation after start-up, or a
 * plugin whose host owns every device buffer.  This entry point runs exactly
 * kda_chunk_fwd with cp_mode = KDA_CP_ON, but takes its scratch (segment
 * table, per-segment transitions M and N, per-segment initial states) from
 * one fixed device array inside the library, KDA_NOALLOC_SCRATCH_BYTES
 * (64 MiB) on every GPU that loads the library, held until the process exits.
 * The caller still passes all inputs and outputs, with kda_chunk_fwd's
 * meaning, layout and rules.
 *
 * Limit: kda_chunk_fwd_workspace_size(N, T, H, dk, dv, KDA_CP_ON, segment_len)
 * must not exceed KDA_NOALLOC_SCRATCH_BYTES (about 3 * segments * H * dk * dv
 * * 4 bytes); larger requests return KDA_ERR_SCRATCH_LIMIT before any launch.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  Every call shares the one array and it keeps the last call's
 * contents (nothing in it needs clearing): calls that overlap on the GPU, on
 * any streams, race on it and must be serialised by the caller.
 */
#define KDA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
int kda_chunk_fwd_cp_noalloc(const void *q, const void *k, const void *v, const float *g,
                             const float *beta, const int32_t *cu_seqlens, int N, int T, int H,
                             int dk, int dv, const float *initial_state, float *final_state,
                             void *o, float scale, float g_min, int in_dtype, int segment_len,
                             uint32_t *status, void *stream);

/*
 * Launch timing, for measurement: between kda_kernel_timing_start() and
 * kda_kernel_timing_stop(), every kernel launch of this library (any thread,
 * any stream) is bracketed by two CUDA events recorded on its stream.  Stop
 * waits for those events and writes, per kernel family k < nkinds (the
 * KDA_KERNEL_* numbers), the launch count launches[k] and the summed device
 * time total_ms[k]; it returns KDA_ERR_CUDA if an event could not be read.
 * Start discards anything recorded before.  Host arithmetic and event calls
 * only; this facility has no counterpart on the pages.
 */
int kda_kernel_timing_start(void);
int kda_kernel_timing_stop(int *launches, float *total_ms, int nkinds);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
