// chunk_bwd.cu -- backward of the prefill on the CUDA cores (sm_103a): dq, dk,
// dv, dg, dbeta and dS0 from the output gradient do and the final-state
// gradient dS_final.
//
// Reverse mode of the token recurrence (the pages name training, which needs
// this pass, as the other use of the chunk kernel: "Noyaux KDA et FlashKDA",
// section "FlashKDA : le noyau par blocs").  Per token, with S the state
// before it, D = Diag(e^{max(g, g_min)}), X = D S, p = X^T k, u = b (v - p),
// S' = X + k u^T, o = scale S'^T q, and G the gradient w.r.t. S' coming from
// later tokens:
//   G += scale q do^T;  dq = scale S' do;  du = G^T k;  dv = b du;
//   db = du . (v - p);  dk = G u - b X du;  dX = G - b k du^T;
//   dg_i = sum_j dX_ij X_ij (zero where g_i < g_min);  G <- D dX.
// The value columns of the state evolve independently (k, g, b are shared by
// all of them).  A group of D threads owns 32 value columns: its thread i
// owns key row i of them (32 fp32 of S and 32 of G in registers, worked as 16
// pairs by the packed f32x2 instructions).  Sums over key rows (p, du) go
// through a 32-lane transpose-sum and the group's warps; sums over value
// columns (dq, dk, dg, db) are per-thread partials added across the groups in
// group order.
//
// Two forms with the same arithmetic in the same order (so the same bits):
//  * whole (SPLIT = false): a CTA of D/32 groups walks one (sequence, head);
//    the column sums meet in shared memory token by token;
//  * split (SPLIT = true): a cluster of D/32 one-group CTAs walks one
//    (sequence, head), so a unit spreads over D/32 SMs.  Every CTA writes its
//    column partials of a chunk to a buffer of its own in global memory, a
//    cluster barrier closes the chunk, and each CTA then adds the partials of
//    all groups for a share of the chunk's tokens.  Two buffers per CTA
//    alternate by chunk, so one barrier per chunk suffices: a CTA starts
//    writing the buffer of chunk c + 2 only after every CTA of the cluster
//    has arrived at the barrier of chunk c + 1, i.e. finished reading chunk c.
// CTAs (clusters) are persistent, at most kBwdMaxCtas units at a time (one
// scratch slot each), and stride over the (sequence, head) units.
// Pass 1 walks the sequence forward, keeps the state at every chunk start
// (64 tokens) in a slot-indexed buffer (chunk j of sequence n is slot
// floor(t0 / 64) + n + j) and w = v - p of every token in a [T][H][d] buffer;
// pass 2 takes the chunks in reverse, recomputes the chunk's states from its
// checkpoint and the stored w (S' = D S + k (b w)^T: the same operations as
// pass 1, so the same bits, without the sum over key rows) into a per-CTA
// scratch and runs the backward steps over them.  Each
// chunk's b and the CTA's value columns of v and do, and its k and g half a
// chunk (32 tokens) at a time, are copied into shared memory by cp.async
// batches (one memory latency per batch); q is read from global memory one
// token ahead, and (split form) the recomputed state of the next token is
// copied into one of two shared-memory buffers while the current token's step
// runs.
// The state blocks that go through global memory (chunk-start states and the
// recomputed per-token states) are stored thread-major: the float4 of value
// columns c .. c + 3 of every thread lie side by side, so each float4 access
// of a warp covers 512 contiguous bytes.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace bw {

constexpr int CH = 64;
constexpr int HC = 32;  // tokens of k and g staged at a time

template <bool BF16>
struct InType;
template <>
struct InType<true> {
    using T = __nv_bfloat16;
};
template <>
struct InType<false> {
    using T = float;
};

template <bool BF16>
__device__ __forceinline__ float ld_in(const void *p, size_t idx) {
    if constexpr (BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[idx]);
    else return reinterpret_cast<const float *>(p)[idx];
}
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
// four consecutive elements of shared memory as two pairs
__device__ __forceinline__ void ld4(const float *p, float2 &a, float2 &b) {
    const float4 v = *reinterpret_cast<const float4 *>(p);
    a = make_float2(v.x, v.y);
    b = make_float2(v.z, v.w);
}
__device__ __forceinline__ void ld4(const __nv_bfloat16 *p, float2 &a, float2 &b) {
    const uint2 v = *reinterpret_cast<const uint2 *>(p);
    a = unpack_bf16(v.x);
    b = unpack_bf16(v.y);
}
__device__ __forceinline__ float2 bc2(float a) { return make_float2(a, a); }

// v[j] summed over the 32 lanes of the warp; lane l returns the sum of column
// l (five exchange rounds of halves, the adds of a round paired; v is
// destroyed)
__device__ __forceinline__ float transpose_sum32(float (&v)[32], int lane) {
#pragma unroll
    for (int w = 16; w >= 2; w >>= 1) {
        const bool hi = (lane & w) != 0;
#pragma unroll
        for (int c = 0; c < w; c += 2) {
            const float s0 = hi ? v[c] : v[c + w], s1 = hi ? v[c + 1] : v[c + 1 + w];
            const float k0 = hi ? v[c + w] : v[c], k1 = hi ? v[c + 1 + w] : v[c + 1];
            const float r0 = __shfl_xor_sync(0xffffffffu, s0, w), r1 = __shfl_xor_sync(0xffffffffu, s1, w);
            const float2 sum = __fadd2_rn(make_float2(k0, k1), make_float2(r0, r1));
            v[c] = sum.x;
            v[c + 1] = sum.y;
        }
    }
    const bool hi = (lane & 1) != 0;
    const float send = hi ? v[0] : v[1], keep = hi ? v[1] : v[0];
    return keep + __shfl_xor_sync(0xffffffffu, send, 1);
}

__device__ __forceinline__ void group_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}

// all threads of all CTAs of the cluster; global writes before it are visible
// to the reads after it in every CTA of the cluster
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// 16-byte global -> shared copies that complete asynchronously (L2 only), the
// fence that closes a batch and the wait for all of this thread's batches
__device__ __forceinline__ void cpa16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cpa4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cpa_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
__device__ __forceinline__ void cpa_wait_all() { asm volatile("cp.async.wait_group 0;\n" ::: "memory"); }

// the float4 of columns c .. c + 3 (c a multiple of 4) of thread tid's slab in
// a thread-major state block of nt threads
__device__ __forceinline__ float4 *slab4(float *blk, int tid, int c, int nt) {
    return reinterpret_cast<float4 *>(blk) + (size_t)(c >> 2) * nt + tid;
}
__device__ __forceinline__ const float4 *slab4(const float *blk, int tid, int c, int nt) {
    return reinterpret_cast<const float4 *>(blk) + (size_t)(c >> 2) * nt + tid;
}
__device__ __forceinline__ void ld_slab(float2 (&S)[16], const float *blk, int tid, int nt) {
#pragma unroll
    for (int c = 0; c < 32; c += 4) {
        const float4 v4 = *slab4(blk, tid, c, nt);
        S[c / 2] = make_float2(v4.x, v4.y);
        S[c / 2 + 1] = make_float2(v4.z, v4.w);
    }
}
// thread tid's slab of a thread-major block, global -> shared, asynchronously
__device__ __forceinline__ void cpa_slab(float *dst, const float *src, int tid, int nt) {
#pragma unroll
    for (int c = 0; c < 32; c += 4) cpa16(slab4(dst, tid, c, nt), slab4(src, tid, c, nt));
}
__device__ __forceinline__ void st_slab(float *blk, const float2 (&S)[16], int tid, int nt) {
#pragma unroll
    for (int c = 0; c < 32; c += 4)
        *slab4(blk, tid, c, nt) = make_float4(S[c / 2].x, S[c / 2].y, S[c / 2 + 1].x, S[c / 2 + 1].y);
}
// 32 consecutive floats of a row of a user [d][d] block (zero when absent)
__device__ __forceinline__ void ld_row32(float2 (&S)[16], const float *src) {
#pragma unroll
    for (int c = 0; c < 32; c += 4) {
        const float4 v4 = src ? *reinterpret_cast<const float4 *>(src + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        S[c / 2] = make_float2(v4.x, v4.y);
        S[c / 2 + 1] = make_float2(v4.z, v4.w);
    }
}

// column partials of one chunk of one CTA: [CH][3][D] (scale dq, dk, dg), then [CH] (db)
template <int D>
__host__ __device__ constexpr size_t part_floats() {
    return (size_t)CH * (3 * D + 1);
}

template <int D, bool BF16, bool SPLIT>
struct BwdSmem {
    using TI = typename InType<BF16>::T;
    static constexpr int NG = SPLIT ? 1 : D / 32;  // groups of the CTA
    static constexpr int VW = 32 * NG;             // value columns of the CTA
    static constexpr int WPG = D / 32;             // warps per group
    static constexpr size_t off_v = 0;                                         // f32 [CH][VW]: w = v - p
    static constexpr size_t off_vr = off_v + (size_t)CH * VW * 4;              // TI [CH][VW]: v
    static constexpr size_t off_do = off_vr + (size_t)CH * VW * sizeof(TI);   // TI [CH][VW]
    static constexpr size_t off_k = off_do + (size_t)CH * VW * sizeof(TI);    // TI [HC][D]
    static constexpr size_t off_g = off_k + (size_t)HC * D * sizeof(TI);      // f32 [HC][D] (raw g)
    static constexpr size_t off_b = off_g + (size_t)HC * D * 4;                // f32 [CH]
    static constexpr size_t off_red = off_b + (size_t)CH * 4;                  // f32 [NG][WPG][32]
    static constexpr size_t off_du = off_red + (size_t)NG * WPG * 32 * 4;      // f32 [VW]
    static constexpr size_t off_row = off_du + (size_t)VW * 4;                 // f32 [3][NG][D] (whole form)
    static constexpr size_t off_db = off_row + (SPLIT ? 0 : (size_t)3 * NG * D * 4);  // f32 [NG]
    static constexpr size_t off_sp = off_db + 64;  // f32 [2][32 D]: next states (split form)
    static constexpr size_t bytes = off_sp + (SPLIT ? (size_t)2 * 32 * D * 4 : 0);
    static_assert(bytes <= 227 * 1024, "shared memory of one CTA");
};

template <int D, bool BF16, bool SPLIT>
__global__ void __launch_bounds__(SPLIT ? D : D * D / 32, SPLIT ? 3 : 1) kda_chunk_bwd_kernel(const BwdArgs p) {
    using L = BwdSmem<D, BF16, SPLIT>;
    using TI = typename L::TI;
    constexpr int NG = L::NG, VW = L::VW, WPG = L::WPG;
    constexpr int NC = SPLIT ? D / 32 : 1;  // CTAs per unit (the cluster)
    constexpr int NT = NG * D;              // threads of the CTA
    extern __shared__ __align__(16) unsigned char smem[];
    float *sV = reinterpret_cast<float *>(smem + L::off_v);
    TI *sVr = reinterpret_cast<TI *>(smem + L::off_vr);
    TI *sDo = reinterpret_cast<TI *>(smem + L::off_do);
    TI *sK = reinterpret_cast<TI *>(smem + L::off_k);
    float *sG = reinterpret_cast<float *>(smem + L::off_g);
    float *sB = reinterpret_cast<float *>(smem + L::off_b);
    float *sRed = reinterpret_cast<float *>(smem + L::off_red);
    float *sDu = reinterpret_cast<float *>(smem + L::off_du);
    float *sRow = reinterpret_cast<float *>(smem + L::off_row);
    float *sDb = reinterpret_cast<float *>(smem + L::off_db);
    float *sSp = reinterpret_cast<float *>(smem + L::off_sp);

    const int tid = threadIdx.x, lane = tid & 31;
    const int gi = tid / D, i = tid % D, wg = i >> 5;     // group in the CTA, key row, warp in the group
    const int rank = SPLIT ? (int)(blockIdx.x % NC) : 0;  // CTA in its cluster (NC consecutive CTAs)
    const int cl = blockIdx.x / NC, ncl = gridDim.x / NC;
    const int cbase = 32 * rank;     // first value column of the CTA
    const int vc = 32 * gi;          // first value column of the thread's group, within the CTA's
    const int c0 = cbase + vc;       // ... and within the state
    const int H = p.H, nunits = p.N * H;
    const size_t DD = (size_t)D * D, BLK = (size_t)32 * NT;  // a unit's state; the CTA's share of it
    const float g_min = p.g_min, scale = p.scale;
    // the CTA's scratch slot: [CH][BLK], its columns of the state before each token of the chunk
    float *scr = p.scratch + (size_t)blockIdx.x * CH * BLK;
    // column partials (split form): two buffers per CTA; CTA s of this cluster owns slot cl * NC + s
    auto part = [&](int s, int buf) { return p.partials + ((size_t)(cl * NC + s) * 2 + buf) * part_floats<D>(); };
    int pbuf = 0;

    for (int un = cl; un < nunits; un += ncl) {
    const int n = un / H, h = un % H;
    const int t0 = p.cu_seqlens[n], t1 = p.cu_seqlens[n + 1];
    if (t0 < 0 || t1 < t0 || t1 > p.T) {  // taken by every CTA of the cluster alike
        if (tid == 0 && h == 0 && rank == 0) report_status(p.status, KDA_STATUS_BAD_SEQLENS);
        continue;
    }
    const int Ln = t1 - t0, nch = (Ln + CH - 1) / CH;
    const size_t unit = (size_t)un;

    // k and g rows of tokens 32 hf .. 32 hf + 31 of chunk j into shared memory
    // (row = token mod 32), as cp.async pieces of 16 bytes
    auto stage_kg = [&](int j, int hf) {
        const int tb = t0 + CH * j + HC * hf, lc = min(HC, t1 - tb);
        constexpr int KP = D * (int)sizeof(TI) / 16, KE = 16 / (int)sizeof(TI), GP = D / 4;
        for (int idx = tid; idx < lc * KP; idx += NT) {
            const int tt = idx / KP, c = (idx % KP) * KE;
            cpa16(sK + tt * D + c, reinterpret_cast<const TI *>(p.k) + ((size_t)(tb + tt) * H + h) * D + c);
        }
        for (int idx = tid; idx < lc * GP; idx += NT) {
            const int tt = idx / GP, c = (idx % GP) * 4;
            cpa16(sG + tt * D + c, p.g + ((size_t)(tb + tt) * H + h) * D + c);
        }
    };
    // the chunk's b and the CTA's columns of v (forward pass) or of the
    // stored w and of do (backward pass) into shared memory, as cp.async pieces
    auto stage = [&](int j, bool bwd) {
        const int tb = t0 + CH * j, lc = min(CH, t1 - tb);
        constexpr int VP = VW * (int)sizeof(TI) / 16, VE = 16 / (int)sizeof(TI), WP = VW / 4;
        for (int idx = tid; idx < lc * VP; idx += NT) {
            const int tt = idx / VP, c = (idx % VP) * VE;
            const size_t th = ((size_t)(tb + tt) * H + h) * D + cbase + c;
            if (bwd) cpa16(sDo + tt * VW + c, reinterpret_cast<const TI *>(p.dout) + th);
            else cpa16(sVr + tt * VW + c, reinterpret_cast<const TI *>(p.v) + th);
        }
        if (bwd)
            for (int idx = tid; idx < lc * WP; idx += NT) {
                const int tt = idx / WP, c = (idx % WP) * 4;
                cpa16(sV + tt * VW + c, p.wbuf + ((size_t)(tb + tt) * H + h) * D + cbase + c);
            }
        for (int tt = tid; tt < lc; tt += NT) cpa4(sB + tt, p.beta + (size_t)(tb + tt) * H + h);
    };
    // wait for this thread's copies, then for every thread's
    auto landed = [&]() {
        cpa_commit();
        cpa_wait_all();
        __syncthreads();
    };
    // one forward step of token tt of the staged chunk on this thread's slab S
    // (row i, columns c0 ..); the token's v row becomes w = v - p (u = b w)
    auto fwd_step = [&](float2 (&S)[16], int tt) {
        const int r = tt & (HC - 1);
        const float e = __expf(fmaxf(sG[r * D + i], g_min));
        const float ki = to_f(sK[r * D + i]), b = sB[tt];
        const float2 e2 = bc2(e), k2 = bc2(ki), b2 = bc2(b);
        float pv[32];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const float2 x = __fmul2_rn(__fmul2_rn(e2, S[c]), k2);
            pv[2 * c] = x.x;
            pv[2 * c + 1] = x.y;
        }
        const float ps = transpose_sum32(pv, lane);
        sRed[(gi * WPG + wg) * 32 + lane] = ps;
        group_sync(1 + gi, D);
        if (wg == 0) {
            float pj = 0.f;
#pragma unroll
            for (int w = 0; w < WPG; ++w) pj += sRed[(gi * WPG + w) * 32 + lane];
            sV[tt * VW + vc + lane] = to_f(sVr[tt * VW + vc + lane]) - pj;
        }
        group_sync(1 + gi, D);
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
            float2 wa, wb;
            ld4(sV + tt * VW + vc + c, wa, wb);
            S[c / 2] = __ffma2_rn(k2, __fmul2_rn(b2, wa), __fmul2_rn(e2, S[c / 2]));
            S[c / 2 + 1] = __ffma2_rn(k2, __fmul2_rn(b2, wb), __fmul2_rn(e2, S[c / 2 + 1]));
        }
    };
    // the same step with w = v - p already staged (pass 2)
    auto rec_step = [&](float2 (&S)[16], int tt) {
        const int r = tt & (HC - 1);
        const float e = __expf(fmaxf(sG[r * D + i], g_min));
        const float ki = to_f(sK[r * D + i]), b = sB[tt];
        const float2 e2 = bc2(e), k2 = bc2(ki), b2 = bc2(b);
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
            float2 wa, wb;
            ld4(sV + tt * VW + vc + c, wa, wb);
            S[c / 2] = __ffma2_rn(k2, __fmul2_rn(b2, wa), __fmul2_rn(e2, S[c / 2]));
            S[c / 2 + 1] = __ffma2_rn(k2, __fmul2_rn(b2, wb), __fmul2_rn(e2, S[c / 2 + 1]));
        }
    };
    auto slot_of = [&](int j) { return (size_t)(t0 / CH + n + j); };
    // the CTA's share of the unit's checkpoint block of chunk j
    auto ckpt_blk = [&](int j) { return p.ckpt + (slot_of(j) * H + h) * DD + (size_t)rank * BLK; };

    // ---------------------------------------------------------------- pass 1: chunk-start states
    {
        float2 S[16];
        ld_row32(S, p.S0 ? p.S0 + unit * DD + (size_t)i * D + c0 : nullptr);
        for (int j = 0; j < nch; ++j) {
            const int tb = t0 + CH * j, lc = min(CH, t1 - tb);
            st_slab(ckpt_blk(j), S, tid, NT);
            stage(j, false);
            for (int hf = 0; HC * hf < lc; ++hf) {
                stage_kg(j, hf);
                landed();
                for (int tt = HC * hf; tt < min(lc, HC * (hf + 1)); ++tt) fwd_step(S, tt);
                __syncthreads();
            }
            // the chunk's w rows (this CTA's columns) to the w buffer
            for (int idx = tid; idx < lc * (VW / 4); idx += NT) {
                const int tt = idx / (VW / 4), c = (idx % (VW / 4)) * 4;
                *reinterpret_cast<float4 *>(p.wbuf + ((size_t)(tb + tt) * H + h) * D + cbase + c) =
                    *reinterpret_cast<const float4 *>(sV + tt * VW + c);
            }
        }
        __syncthreads();  // sV is restaged next
    }

    // ---------------------------------------------------------------- pass 2: chunks in reverse
    float2 G[16];
    ld_row32(G, p.dS_final ? p.dS_final + unit * DD + (size_t)i * D + c0 : nullptr);
    for (int j = nch - 1; j >= 0; --j) {
        const int tb = t0 + CH * j, lc = min(CH, t1 - tb);
        stage(j, true);
        // recompute the chunk's states from the stored w (the one before each
        // token goes to the scratch); k and g of the chunk's last half stay staged
        {
            float2 S[16];
            ld_slab(S, ckpt_blk(j), tid, NT);
            for (int hf = 0; HC * hf < lc; ++hf) {
                if (hf) __syncthreads();
                stage_kg(j, hf);
                landed();
                for (int tt = HC * hf; tt < min(lc, HC * (hf + 1)); ++tt) {
                    st_slab(scr + (size_t)tt * BLK, S, tid, NT);
                    rec_step(S, tt);
                }
            }
        }
        // backward steps, last token first, with q one token ahead in a register
        float q_next = ld_in<BF16>(p.q, ((size_t)(tb + lc - 1) * H + h) * D + i);
        float *pw = SPLIT ? part(rank, pbuf) : nullptr;
        // split form: token tt's state goes through buffer tt & 1; a buffer is
        // refilled one step after the step that read it, whose arithmetic has
        // consumed the values (so the read is complete)
        if constexpr (SPLIT) {
            cpa_slab(sSp + (size_t)((lc - 1) & 1) * BLK, scr + (size_t)(lc - 1) * BLK, tid, NT);
            cpa_commit();
        }
        for (int tt = lc - 1; tt >= 0; --tt) {
            const size_t th = (size_t)(tb + tt) * H + h;
            if (tt == HC - 1 && lc > HC) {  // into the chunk's first half: its k and g
                __syncthreads();
                stage_kg(j, 0);
                landed();
            }
            const float qi = q_next;
            if (tt > 0) q_next = ld_in<BF16>(p.q, (th - H) * D + i);
            const int r = tt & (HC - 1);
            const float graw = sG[r * D + i];
            const float e = __expf(fmaxf(graw, g_min));
            const float ki = to_f(sK[r * D + i]);
            const float b = sB[tt];
            const float2 e2 = bc2(e), k2 = bc2(ki), b2 = bc2(b);
            float2 Sp[16];
            if constexpr (SPLIT) {
                cpa_wait_all();
                ld_slab(Sp, sSp + (size_t)(tt & 1) * BLK, tid, NT);
                if (tt > 0) {
                    cpa_slab(sSp + (size_t)((tt - 1) & 1) * BLK, scr + (size_t)(tt - 1) * BLK, tid, NT);
                    cpa_commit();
                }
            } else {
                ld_slab(Sp, scr + (size_t)tt * BLK, tid, NT);
            }
            // G += scale q do^T; dq partial = scale S' do over this group's columns
            float2 dq2 = make_float2(0.f, 0.f);
            float gk[32];
            const float2 sq2 = bc2(scale * qi);
            const TI *dorow = sDo + tt * VW + vc;
            const float *wrow = sV + tt * VW + vc;  // 16-byte aligned
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
                float2 d2[2], w2[2];
                ld4(dorow + c, d2[0], d2[1]);
                ld4(wrow + c, w2[0], w2[1]);
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    const int cc = c / 2 + m;
                    const float2 st = __ffma2_rn(k2, __fmul2_rn(b2, w2[m]), __fmul2_rn(e2, Sp[cc]));  // S' = X + k u^T
                    dq2 = __ffma2_rn(st, d2[m], dq2);
                    G[cc] = __ffma2_rn(sq2, d2[m], G[cc]);
                    const float2 x = __fmul2_rn(G[cc], k2);
                    gk[2 * cc] = x.x;
                    gk[2 * cc + 1] = x.y;
                }
            }
            const float dus = transpose_sum32(gk, lane);
            sRed[(gi * WPG + wg) * 32 + lane] = dus;
            group_sync(1 + gi, D);
            if (wg == 0) {
                float du = 0.f;
#pragma unroll
                for (int w = 0; w < WPG; ++w) du += sRed[(gi * WPG + w) * 32 + lane];
                sDu[vc + lane] = du;
                p.dv[th * D + c0 + lane] = b * du;
                float term = du * sV[tt * VW + vc + lane];  // du (v - p)
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) term += __shfl_xor_sync(0xffffffffu, term, o);
                if (lane == 0) {
                    if constexpr (SPLIT) pw[(size_t)CH * 3 * D + tt] = term;
                    else sDb[gi] = term;
                }
            }
            group_sync(1 + gi, D);
            float2 dk2 = make_float2(0.f, 0.f), dg2 = make_float2(0.f, 0.f);
            const float2 nb2 = bc2(-b), nbk2 = bc2(-(b * ki));
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
                float2 du2[2], w2[2];
                ld4(sDu + vc + c, du2[0], du2[1]);
                ld4(wrow + c, w2[0], w2[1]);
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    const int cc = c / 2 + m;
                    const float2 u = __fmul2_rn(b2, w2[m]);
                    const float2 x = __fmul2_rn(e2, Sp[cc]);
                    dk2 = __ffma2_rn(G[cc], u, dk2);
                    dk2 = __ffma2_rn(__fmul2_rn(nb2, x), du2[m], dk2);
                    const float2 dx = __ffma2_rn(nbk2, du2[m], G[cc]);
                    dg2 = __ffma2_rn(dx, x, dg2);
                    G[cc] = __fmul2_rn(e2, dx);
                }
            }
            const float dqp = scale * (dq2.x + dq2.y), dkp = dk2.x + dk2.y, dgp = dg2.x + dg2.y;
            if constexpr (SPLIT) {
                float *pr = pw + (size_t)tt * 3 * D;
                pr[i] = dqp;
                pr[D + i] = dkp;
                pr[2 * D + i] = dgp;
            } else {
                sRow[(0 * NG + gi) * D + i] = dqp;
                sRow[(1 * NG + gi) * D + i] = dkp;
                sRow[(2 * NG + gi) * D + i] = dgp;
                __syncthreads();
                if (gi == 0) {
                    float a0 = 0.f, a1 = 0.f, a2 = 0.f;
#pragma unroll
                    for (int gg = 0; gg < NG; ++gg) {
                        a0 += sRow[(0 * NG + gg) * D + i];
                        a1 += sRow[(1 * NG + gg) * D + i];
                        a2 += sRow[(2 * NG + gg) * D + i];
                    }
                    p.dq[th * D + i] = a0;
                    p.dk[th * D + i] = a1;
                    p.dg[th * D + i] = (graw < g_min) ? 0.f : a2;
                }
                if (tid == 0) {
                    float s = 0.f;
#pragma unroll
                    for (int gg = 0; gg < NG; ++gg) s += sDb[gg];
                    p.dbeta[th] = s;
                }
                __syncthreads();
            }
        }
        if constexpr (SPLIT) {
            // the chunk's column partials of every CTA of the cluster, added in
            // group order, for the tokens rank, rank + NC, ... of the chunk
            cluster_sync();
            // four tokens at a time: all their partials are loaded before any sum
            for (int tq = rank; tq < lc; tq += 4 * NC) {
                float v[4][NC][3], vb[4][NC];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int tt = tq + u * NC;
#pragma unroll
                    for (int s = 0; s < NC; ++s) {
                        const float *pr = part(s, pbuf);
                        const bool ok = tt < lc;
#pragma unroll
                        for (int x = 0; x < 3; ++x) v[u][s][x] = ok ? __ldcg(pr + (size_t)tt * 3 * D + x * D + i) : 0.f;
                        vb[u][s] = (ok && tid == 0) ? __ldcg(pr + (size_t)CH * 3 * D + tt) : 0.f;
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int tt = tq + u * NC;
                    if (tt >= lc) break;
                    const size_t th = (size_t)(tb + tt) * H + h;
                    float a0 = 0.f, a1 = 0.f, a2 = 0.f, sb = 0.f;
#pragma unroll
                    for (int s = 0; s < NC; ++s) {
                        a0 += v[u][s][0];
                        a1 += v[u][s][1];
                        a2 += v[u][s][2];
                        sb += vb[u][s];
                    }
                    p.dq[th * D + i] = a0;
                    p.dk[th * D + i] = a1;
                    p.dg[th * D + i] = (p.g[th * D + i] < g_min) ? 0.f : a2;
                    if (tid == 0) p.dbeta[th] = sb;
                }
            }
            pbuf ^= 1;
        }
    }
    if (p.dS0) {
        float *dst = p.dS0 + unit * DD + (size_t)i * D + c0;
#pragma unroll
        for (int c = 0; c < 32; c += 4)
            *reinterpret_cast<float4 *>(dst + c) = make_float4(G[c / 2].x, G[c / 2].y, G[c / 2 + 1].x, G[c / 2 + 1].y);
    }
    __syncthreads();  // the next unit stages into the same shared memory
    }  // units
}

template <int D, bool BF16, bool SPLIT>
static cudaError_t launch_t(const BwdArgs &a, cudaStream_t st) {
    using L = BwdSmem<D, BF16, SPLIT>;
    auto kern = kda_chunk_bwd_kernel<D, BF16, SPLIT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::bytes);
    if (e != cudaSuccess) return e;
    const long units = (long)a.N * a.H;
    int nclusters = (int)(units < kBwdMaxCtas ? units : kBwdMaxCtas);  // units in flight (scratch slots)
    constexpr int NC = SPLIT ? D / 32 : 1;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.blockDim = dim3(SPLIT ? D : D * D / 32);
    cfg.dynamicSmemBytes = L::bytes;
    cfg.stream = st;
    cfg.gridDim = dim3(nclusters * NC);
    if constexpr (SPLIT) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = NC;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int active = 0;
        e = cudaOccupancyMaxActiveClusters(&active, kern, &cfg);
        if (e != cudaSuccess) return e;
        if (active < 1) return launch_t<D, BF16, false>(a, st);  // no cluster fits: one CTA per unit
        if (active < nclusters) nclusters = active;  // the clusters stride over the units
        cfg.gridDim = dim3(nclusters * NC);
    }
    return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace bw

size_t chunk_bwd_partial_floats(int d) { return d == 128 ? bw::part_floats<128>() : bw::part_floats<64>(); }

cudaError_t launch_chunk_bwd(const BwdArgs &a, int d, bool bf16, cudaStream_t st) {
    if (a.N <= 0) return cudaSuccess;
    // the split form unless the caller gave no partial buffers (or, inside
    // launch_t, no cluster of it fits the device)
    const bool split = a.partials != nullptr;
    if (d == 128) {
        if (split) return bf16 ? bw::launch_t<128, true, true>(a, st) : bw::launch_t<128, false, true>(a, st);
        return bf16 ? bw::launch_t<128, true, false>(a, st) : bw::launch_t<128, false, false>(a, st);
    }
    if (d == 64) {
        if (split) return bf16 ? bw::launch_t<64, true, true>(a, st) : bw::launch_t<64, false, true>(a, st);
        return bf16 ? bw::launch_t<64, true, false>(a, st) : bw::launch_t<64, false, false>(a, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace kda
