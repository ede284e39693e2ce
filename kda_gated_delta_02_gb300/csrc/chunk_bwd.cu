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
// all of them), so a CTA of D/32 groups of D threads walks one (sequence,
// head): group c owns value columns 32c .. 32c + 31 and its thread i owns key
// row i of them (32 fp32 of S and 32 of G in registers).  Sums over key rows
// (p, du) go through a 32-lane transpose-sum and the group's warps; sums over
// value columns (dq, dk, dg, db) are per-thread partials added across the
// groups in shared memory, in a fixed order.
// The CTAs are persistent (at most kBwdMaxCtas, one scratch slot each) and
// stride over the (sequence, head) units.
// Pass 1 walks the sequence forward and keeps the state at every chunk start
// (64 tokens) in a slot-indexed buffer (chunk j of sequence n is slot
// floor(t0 / 64) + n + j); pass 2 takes the chunks in reverse, recomputes the
// chunk's states from its checkpoint into a per-CTA scratch (and v - p per
// token in shared memory) and runs the backward steps over them.  Each chunk's
// rows of q, k, v, g, b and do are staged in shared memory first.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace bw {

constexpr int CH = 64;

template <bool BF16>
__device__ __forceinline__ float ld_in(const void *p, size_t idx) {
    if constexpr (BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[idx]);
    else return reinterpret_cast<const float *>(p)[idx];
}

// v[j] summed over the 32 lanes of the warp; lane l returns the sum of column
// l (five exchange rounds of halves; v is destroyed)
__device__ __forceinline__ float transpose_sum32(float (&v)[32], int lane) {
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) {
        const bool hi = (lane & w) != 0;
#pragma unroll
        for (int c = 0; c < w; ++c) {
            const float send = hi ? v[c] : v[c + w];
            const float keep = hi ? v[c + w] : v[c];
            v[c] = keep + __shfl_xor_sync(0xffffffffu, send, w);
        }
    }
    return v[0];
}

__device__ __forceinline__ void group_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(nthreads) : "memory");
}

template <int D>
struct BwdSmem {
    static constexpr int NG = D / 32;
    static constexpr int WPG = D / 32;  // warps per group
    // the chunk's rows, staged once per chunk: v (overwritten by w = v - p as
    // each token's p is formed; u = b w), do, q, k, g (raw) and b
    static constexpr size_t off_v = 0;                                   // f32 [CH][D]
    static constexpr size_t off_do = off_v + (size_t)CH * D * 4;         // f32 [CH][D]
    static constexpr size_t off_q = off_do + (size_t)CH * D * 4;         // f32 [CH][D]
    static constexpr size_t off_k = off_q + (size_t)CH * D * 4;          // f32 [CH][D]
    static constexpr size_t off_g = off_k + (size_t)CH * D * 4;          // f32 [CH][D]
    static constexpr size_t off_b = off_g + (size_t)CH * D * 4;          // f32 [CH]
    static constexpr size_t off_red = off_b + (size_t)CH * 4;            // f32 [NG][WPG][32]
    static constexpr size_t off_du = off_red + (size_t)NG * WPG * 32 * 4;  // f32 [D]
    static constexpr size_t off_row = off_du + (size_t)D * 4;            // f32 [3][NG][D]
    static constexpr size_t off_db = off_row + (size_t)3 * NG * D * 4;   // f32 [NG]
    static constexpr size_t bytes = off_db + 64;
};

template <int D, bool BF16>
__global__ void __launch_bounds__(D * D / 32, 1) kda_chunk_bwd_kernel(const BwdArgs p) {
    using L = BwdSmem<D>;
    constexpr int NG = L::NG, WPG = L::WPG;
    extern __shared__ __align__(16) unsigned char smem[];
    float *sV = reinterpret_cast<float *>(smem + L::off_v);
    float *sDo = reinterpret_cast<float *>(smem + L::off_do);
    float *sQ = reinterpret_cast<float *>(smem + L::off_q);
    float *sK = reinterpret_cast<float *>(smem + L::off_k);
    float *sG = reinterpret_cast<float *>(smem + L::off_g);
    float *sB = reinterpret_cast<float *>(smem + L::off_b);
    float *sRed = reinterpret_cast<float *>(smem + L::off_red);
    float *sDu = reinterpret_cast<float *>(smem + L::off_du);
    float *sRow = reinterpret_cast<float *>(smem + L::off_row);
    float *sDb = reinterpret_cast<float *>(smem + L::off_db);

    const int tid = threadIdx.x, lane = tid & 31;
    const int gi = tid / D, i = tid % D, wg = i >> 5;  // group, key row, warp in the group
    const int c0 = 32 * gi;                            // first value column of the group
    const int H = p.H, nunits = p.N * H;
    const size_t DD = (size_t)D * D;
    const float g_min = p.g_min, scale = p.scale;
    // this CTA's scratch slot: [CH][D][D], the state before each token of the chunk
    float *scr = p.scratch + (size_t)blockIdx.x * CH * DD;
    // persistent: units (sequence, head) strided over the CTAs
    for (int un = blockIdx.x; un < nunits; un += gridDim.x) {
    const int n = un / H, h = un % H;
    const int t0 = p.cu_seqlens[n], t1 = p.cu_seqlens[n + 1];
    if (t0 < 0 || t1 < t0 || t1 > p.T) {
        if (tid == 0 && h == 0) report_status(p.status, KDA_STATUS_BAD_SEQLENS);
        continue;
    }
    const int Ln = t1 - t0, nch = (Ln + CH - 1) / CH;
    const size_t unit = (size_t)un;

    // the rows of chunk j (tokens t0 + 64 j ..) into shared memory; q and do
    // only for the backward pass
    auto stage = [&](int j, bool bwd) {
        const int tb = t0 + CH * j, lc = min(CH, t1 - tb);
        for (int idx = tid; idx < lc * D; idx += NG * D) {
            const int tt = idx / D, c = idx % D;
            const size_t th = ((size_t)(tb + tt) * H + h) * D + c;
            sV[tt * D + c] = ld_in<BF16>(p.v, th);
            sK[tt * D + c] = ld_in<BF16>(p.k, th);
            sG[tt * D + c] = p.g[th];
            if (bwd) {
                sDo[tt * D + c] = ld_in<BF16>(p.dout, th);
                sQ[tt * D + c] = ld_in<BF16>(p.q, th);
            }
        }
        for (int tt = tid; tt < lc; tt += NG * D) sB[tt] = p.beta[(size_t)(tb + tt) * H + h];
    };
    // one forward step of token tt of the staged chunk on this thread's slab S
    // (row i, columns c0 ..); the token's v row becomes w = v - p (u = b w)
    auto fwd_step = [&](float (&S)[32], int tt) {
        const float e = __expf(fmaxf(sG[tt * D + i], g_min));
        const float ki = sK[tt * D + i], b = sB[tt];
        float pv[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) pv[c] = (e * S[c]) * ki;
        const float ps = transpose_sum32(pv, lane);
        sRed[(gi * WPG + wg) * 32 + lane] = ps;
        group_sync(1 + gi, D);
        if (wg == 0) {
            float pj = 0.f;
#pragma unroll
            for (int w = 0; w < WPG; ++w) pj += sRed[(gi * WPG + w) * 32 + lane];
            sV[tt * D + c0 + lane] -= pj;
        }
        group_sync(1 + gi, D);
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
            const float4 w4 = *reinterpret_cast<const float4 *>(sV + tt * D + c0 + c);
            S[c + 0] = fmaf(ki, b * w4.x, e * S[c + 0]);
            S[c + 1] = fmaf(ki, b * w4.y, e * S[c + 1]);
            S[c + 2] = fmaf(ki, b * w4.z, e * S[c + 2]);
            S[c + 3] = fmaf(ki, b * w4.w, e * S[c + 3]);
        }
    };
    auto slot_of = [&](int j) { return (size_t)(t0 / CH + n + j); };

    // ---------------------------------------------------------------- pass 1: chunk-start states
    {
        float S[32];
        const float *src = p.S0 ? p.S0 + unit * DD + (size_t)i * D + c0 : nullptr;
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
            const float4 v4 = src ? *reinterpret_cast<const float4 *>(src + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            S[c] = v4.x;
            S[c + 1] = v4.y;
            S[c + 2] = v4.z;
            S[c + 3] = v4.w;
        }
        for (int j = 0; j < nch; ++j) {
            float *ck = p.ckpt + (slot_of(j) * H + h) * DD + (size_t)i * D + c0;
#pragma unroll
            for (int c = 0; c < 32; c += 4)
                *reinterpret_cast<float4 *>(ck + c) = make_float4(S[c], S[c + 1], S[c + 2], S[c + 3]);
            if (j == nch - 1) break;  // the last chunk's states are recomputed in pass 2
            stage(j, false);
            __syncthreads();
            for (int tt = 0; tt < CH; ++tt) fwd_step(S, tt);
            __syncthreads();
        }
    }

    // ---------------------------------------------------------------- pass 2: chunks in reverse
    float G[32];
    {
        const float *src = p.dS_final ? p.dS_final + unit * DD + (size_t)i * D + c0 : nullptr;
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
            const float4 v4 = src ? *reinterpret_cast<const float4 *>(src + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            G[c] = v4.x;
            G[c + 1] = v4.y;
            G[c + 2] = v4.z;
            G[c + 3] = v4.w;
        }
    }
    for (int j = nch - 1; j >= 0; --j) {
        const int tb = t0 + CH * j, lc = min(CH, t1 - tb);
        stage(j, true);
        __syncthreads();
        // recompute the chunk's states (the one before each token goes to the scratch)
        {
            float S[32];
            const float *ck = p.ckpt + (slot_of(j) * H + h) * DD + (size_t)i * D + c0;
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
                const float4 v4 = *reinterpret_cast<const float4 *>(ck + c);
                S[c] = v4.x;
                S[c + 1] = v4.y;
                S[c + 2] = v4.z;
                S[c + 3] = v4.w;
            }
            for (int tt = 0; tt < lc; ++tt) {
                float *dst = scr + (size_t)tt * DD + (size_t)i * D + c0;
#pragma unroll
                for (int c = 0; c < 32; c += 4)
                    *reinterpret_cast<float4 *>(dst + c) = make_float4(S[c], S[c + 1], S[c + 2], S[c + 3]);
                fwd_step(S, tt);
            }
        }
        // backward steps, last token first; the state of the token four steps
        // on is brought into L2 while this one runs
        constexpr int PF = 4;
        for (int tt = lc - 1; tt >= lc - PF && tt >= 0; --tt)
            asm volatile("prefetch.global.L2 [%0];\n" ::"l"(scr + (size_t)tt * DD + (size_t)i * D + c0));
        for (int tt = lc - 1; tt >= 0; --tt) {
            const size_t th = (size_t)(tb + tt) * H + h;
            if (tt >= PF)
                asm volatile("prefetch.global.L2 [%0];\n" ::"l"(scr + (size_t)(tt - PF) * DD + (size_t)i * D + c0));
            const float graw = sG[tt * D + i];
            const float e = __expf(fmaxf(graw, g_min));
            const float ki = sK[tt * D + i], qi = sQ[tt * D + i];
            const float b = sB[tt];
            float Sp[32];
            {
                const float *src = scr + (size_t)tt * DD + (size_t)i * D + c0;
#pragma unroll
                for (int c = 0; c < 32; c += 4) {
                    const float4 v4 = *reinterpret_cast<const float4 *>(src + c);
                    Sp[c] = v4.x;
                    Sp[c + 1] = v4.y;
                    Sp[c + 2] = v4.z;
                    Sp[c + 3] = v4.w;
                }
            }
            // G += scale q do^T; dq partial = scale S' do over this group's columns
            float dqp = 0.f, gk[32];
            const float sq = scale * qi;
            const float *dorow = sDo + tt * D + c0, *wrow = sV + tt * D + c0;  // 16-byte aligned
#pragma unroll
            for (int c4 = 0; c4 < 32; c4 += 4) {
                const float4 d4 = *reinterpret_cast<const float4 *>(dorow + c4);
                const float4 w4 = *reinterpret_cast<const float4 *>(wrow + c4);
                const float dd[4] = {d4.x, d4.y, d4.z, d4.w}, ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int c = c4 + m;
                    const float st = fmaf(ki, b * ww[m], e * Sp[c]);  // S' = X + k u^T
                    dqp = fmaf(st, dd[m], dqp);
                    G[c] = fmaf(sq, dd[m], G[c]);
                    gk[c] = G[c] * ki;
                }
            }
            const float dus = transpose_sum32(gk, lane);
            sRed[(gi * WPG + wg) * 32 + lane] = dus;
            group_sync(1 + gi, D);
            if (wg == 0) {
                float du = 0.f;
#pragma unroll
                for (int w = 0; w < WPG; ++w) du += sRed[(gi * WPG + w) * 32 + lane];
                sDu[c0 + lane] = du;
                p.dv[th * D + c0 + lane] = b * du;
                float term = du * sV[tt * D + c0 + lane];  // du (v - p)
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) term += __shfl_xor_sync(0xffffffffu, term, o);
                if (lane == 0) sDb[gi] = term;
            }
            group_sync(1 + gi, D);
            float dkp = 0.f, dgp = 0.f;
            const float bk = b * ki;
#pragma unroll
            for (int c4 = 0; c4 < 32; c4 += 4) {
                const float4 du4 = *reinterpret_cast<const float4 *>(sDu + c0 + c4);
                const float4 w4 = *reinterpret_cast<const float4 *>(wrow + c4);
                const float dus4[4] = {du4.x, du4.y, du4.z, du4.w}, ww[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int c = c4 + m;
                    const float du = dus4[m], u = b * ww[m];
                    const float x = e * Sp[c];
                    dkp = fmaf(G[c], u, dkp);
                    dkp = fmaf(-b * x, du, dkp);
                    const float dx = fmaf(-bk, du, G[c]);
                    dgp = fmaf(dx, x, dgp);
                    G[c] = e * dx;
                }
            }
            sRow[(0 * NG + gi) * D + i] = scale * dqp;
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
    if (p.dS0) {
        float *dst = p.dS0 + unit * DD + (size_t)i * D + c0;
#pragma unroll
        for (int c = 0; c < 32; c += 4) *reinterpret_cast<float4 *>(dst + c) = make_float4(G[c], G[c + 1], G[c + 2], G[c + 3]);
    }
    __syncthreads();  // the next unit stages into the same shared memory
    }  // units
}

template <int D, bool BF16>
static cudaError_t launch_t(const BwdArgs &a, cudaStream_t st) {
    using L = BwdSmem<D>;
    auto kern = kda_chunk_bwd_kernel<D, BF16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::bytes);
    if (e != cudaSuccess) return e;
    const long units = (long)a.N * a.H;
    const int grid = (int)(units < kBwdMaxCtas ? units : kBwdMaxCtas);
    kern<<<grid, D * D / 32, L::bytes, st>>>(a);
    return cudaGetLastError();
}

}  // namespace bw

cudaError_t launch_chunk_bwd(const BwdArgs &a, int d, bool bf16, cudaStream_t st) {
    if (a.N <= 0) return cudaSuccess;
    if (d == 128) return bf16 ? bw::launch_t<128, true>(a, st) : bw::launch_t<128, false>(a, st);
    if (d == 64) return bf16 ? bw::launch_t<64, true>(a, st) : bw::launch_t<64, false>(a, st);
    return cudaErrorInvalidValue;
}

}  // namespace kda
