// decode_verify.cu -- fused speculative-decode verify with replay, sm_103a.
//
// "Noyaux d'inference", section 1 "Le decodage KDA": only the projected inputs
// of draft tokens are cached; the accepted prefix is replayed on chip, and one
// kernel runs short conv -> input norm -> gating -> recurrence -> output norm
// over the replayed tokens, the bonus token and the next draft window, writing
// back the state reached after the bonus token (no per-draft snapshots).
//
// One CTA (D threads, D/32 warps) owns one (request, head).  The a + 1 + Wd
// <= 16 tokens of a request form one 16-row tile, so the replay is the chunk
// (WY) form of the recurrence on a single tile, on the tensor cores:
//   x_t = prod_{r<=t} e^{g_r} (per channel, from the window start; >= e^{-80})
//   A[t,s] = b_t sum_c (k_tc x_tc)(k_sc / x_sc)   (s < t),   T = (I + A)^{-1}
//   B[t,s] =     sum_c (q_tc x_tc)(k_sc / x_sc)   (s <= t)
//   W = T diag(b)(K . x),  U = T diag(b) V - W S0
//   O = scale ((Q . x) S0 + B U)  -> per-head RMSNorm over dv
//   S_a = Diag(x_a) S0 + sum_{s<=a} (k_s . x_a / x_s) u_s^T   (written back)
// The state is read once as bf16, kept exact as a bf16 MMA operand, and the
// written-back state is accumulated in fp32 and rounded once (nearest even).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

constexpr int VT = 16;  // token tile

template <int D>
struct VerifySmem {
    static constexpr int LDS = D + 8;
    static constexpr int CH3 = 3 * D;
    static constexpr int LDR = CH3 + 8;
    static constexpr int MAXROWS = 3 + VT;
    static constexpr int TILE = VT * LDS * 2;  // one [16][D] bf16 plane
    static constexpr int off_s = 0;
    static constexpr int off_u1 = off_s + D * LDS * 2;  // raw rows + raw g | QX KX KR (hi, lo)
    static constexpr int raw_bytes = MAXROWS * LDR * 2 + TILE;
    static constexpr int ops_bytes = 6 * TILE;
    static constexpr int u1_bytes = raw_bytes > ops_bytes ? raw_bytes : ops_bytes;
    static constexpr int off_kt = off_u1 + ((u1_bytes + 127) / 128) * 128;  // K~ hi, lo
    static constexpr int off_v = off_kt + 2 * TILE;                          // V hi, lo
    static constexpr int off_w = off_v + 2 * TILE;
    static constexpr int off_u = off_w + TILE;                               // U hi, lo
    static constexpr int off_af = off_u + 2 * TILE;          // fp32 [16][20]
    static constexpr int off_tf = off_af + VT * 20 * 4;      // fp32 [16][20]
    static constexpr int off_bm = off_tf + VT * 20 * 4;      // bf16 [16][24] hi, lo
    static constexpr int off_beta = off_bm + 2 * VT * 24 * 2; // fp32 [16]
    static constexpr int off_rq = off_beta + VT * 4;         // fp32 [16]
    static constexpr int off_rk = off_rq + VT * 4;           // fp32 [16]
    static constexpr int off_xa = off_rk + VT * 4;           // fp32 [D]
    static constexpr int off_part = off_xa + D * 4;          // fp32 [2][D/32][32]
    static constexpr int bytes = off_part + 2 * (D / 32) * 32 * 4;
};

// x = hi + lo with both halves bf16: products of split operands recover ~16
// mantissa bits (hi*hi + hi*lo + lo*hi), used where bf16 rounding of a
// derived operand would dominate the error.
__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16 &hi, __nv_bfloat16 &lo) {
    hi = __float2bfloat16_rn(x);
    lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}
__device__ __forceinline__ void split_pack(float a, float b, uint32_t &hi, uint32_t &lo) {
    __nv_bfloat16 ha, la, hb, lb;
    split_bf16(a, ha, la);
    split_bf16(b, hb, lb);
    __nv_bfloat162 h2(ha, hb), l2(la, lb);
    hi = *reinterpret_cast<uint32_t *>(&h2);
    lo = *reinterpret_cast<uint32_t *>(&l2);
}

template <int D>
__global__ void __launch_bounds__(D) kda_verify_kernel(VerifyArgs p) {
    using L = VerifySmem<D>;
    constexpr int LDS = L::LDS, LDR = L::LDR, NW = D / 32;
    extern __shared__ __align__(128) unsigned char smem[];
    __nv_bfloat16 *sS = reinterpret_cast<__nv_bfloat16 *>(smem + L::off_s);
    __nv_bfloat16 *sRaw = reinterpret_cast<__nv_bfloat16 *>(smem + L::off_u1);
    __nv_bfloat16 *sGr = sRaw + L::MAXROWS * LDR;
    constexpr int PL = VT * LDS;  // elements in one [16][D] plane
    __nv_bfloat16 *sQX = reinterpret_cast<__nv_bfloat16 *>(smem + L::off_u1);  // hi; lo at +PL
    __nv_bfloat16 *sKX = sQX + 2 * PL;
    __nv_bfloat16 *sKR = sKX + 2 * PL;
    __nv_bfloat16 *sKT = reinterpret_cast<__nv_bfloat16 *>(smem + L::off_kt);
    __nv_bfloat16 *sVv = reinterpret_cast<__nv_bfloat16 *>(smem + L::off_v);
    __nv_bfloat16 *sW = reinterpret_cast<__nv_bfloat16 *>(smem + L::off_w);
    __nv_bfloat16 *sU = reinterpret_cast<__nv_bfloat16 *>(smem + L::off_u);
    float *sAf = reinterpret_cast<float *>(smem + L::off_af);
    float *sTf = reinterpret_cast<float *>(smem + L::off_tf);
    __nv_bfloat16 *sBm = reinterpret_cast<__nv_bfloat16 *>(smem + L::off_bm);
    float *sBeta = reinterpret_cast<float *>(smem + L::off_beta);
    float *sRq = reinterpret_cast<float *>(smem + L::off_rq);
    float *sRk = reinterpret_cast<float *>(smem + L::off_rk);
    float *sXa = reinterpret_cast<float *>(smem + L::off_xa);
    float *sPart = reinterpret_cast<float *>(smem + L::off_part);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, q4 = lane & 3;
    const int H = p.H, W = p.W, Wd = p.Wd;
    const int h = blockIdx.x % H;
    const int r = blockIdx.x / H;
    const int a = p.accepted[r];
    if (a < 0 || a > Wd) {
        if (tid == 0 && h == 0) report_status(p.status, KDA_STATUS_BAD_ACCEPTED_LEN);
        return;
    }
    const int dr = p.draft_len ? p.draft_len[r] : Wd;  // this request's drafts (ragged batches)
    if (dr < 0 || dr > Wd) {
        if (tid == 0 && h == 0) report_status(p.status, KDA_STATUS_BAD_DRAFT_LEN);
        return;
    }
    const int ntok = a + 1 + dr;  // <= 16 (host-checked Wd <= 7)
    const int nrows = (W - 1) + ntok;
    const size_t Cq = (size_t)H * 3 * D;

    const __nv_bfloat16 *tail_g = reinterpret_cast<const __nv_bfloat16 *>(p.tail);
    const __nv_bfloat16 *cq = reinterpret_cast<const __nv_bfloat16 *>(p.cached_qkv);
    const __nv_bfloat16 *nq = reinterpret_cast<const __nv_bfloat16 *>(p.new_qkv);
    const __nv_bfloat16 *cgp = reinterpret_cast<const __nv_bfloat16 *>(p.cached_g);
    const __nv_bfloat16 *ngp = reinterpret_cast<const __nv_bfloat16 *>(p.new_g);
    const __nv_bfloat16 *cbp = reinterpret_cast<const __nv_bfloat16 *>(p.cached_b);
    const __nv_bfloat16 *nbp = reinterpret_cast<const __nv_bfloat16 *>(p.new_b);
    __nv_bfloat16 *stg = reinterpret_cast<__nv_bfloat16 *>(p.state) + ((size_t)r * H + h) * D * D;

    // ---------------------------------------------------------------- loads
    constexpr int RP = D / 8;  // 16-byte pieces per D-wide row segment
    for (int idx = tid; idx < D * RP; idx += D) {
        int row = idx / RP, c = idx % RP;
        cp_async16(&sS[row * LDS + c * 8], stg + (size_t)row * D + c * 8, true);
    }
    for (int idx = tid; idx < nrows * 3 * RP; idx += D) {
        int pr = idx / (3 * RP), rem = idx % (3 * RP), part = rem / RP, c = rem % RP;
        const __nv_bfloat16 *rowp;
        if (pr < W - 1) rowp = tail_g + ((size_t)r * (W - 1) + pr) * Cq;
        else if (pr - (W - 1) < a) rowp = cq + ((size_t)r * Wd + (pr - (W - 1))) * Cq;
        else rowp = nq + ((size_t)r * (Wd + 1) + (pr - (W - 1) - a)) * Cq;
        size_t choff = (size_t)part * H * D + (size_t)h * D + c * 8;
        cp_async16(&sRaw[pr * LDR + part * D + c * 8], rowp + choff, true);
    }
    for (int idx = tid; idx < ntok * RP; idx += D) {
        int t = idx / RP, c = idx % RP;
        const __nv_bfloat16 *src = (t < a) ? cgp + ((size_t)r * Wd + t) * H * D
                                           : ngp + ((size_t)r * (Wd + 1) + (t - a)) * H * D;
        cp_async16(&sGr[t * LDS + c * 8], src + (size_t)h * D + c * 8, true);
    }
    cp_async_commit();
    float braw = 0.f;
    if (tid < ntok) {
        const __nv_bfloat16 *src = (tid < a) ? cbp + ((size_t)r * Wd + tid) * H
                                             : nbp + ((size_t)r * (Wd + 1) + (tid - a)) * H;
        braw = __bfloat162float(src[h]);
    }
    cp_async_wait_all();
    __syncthreads();

    // conv tail write-back: the W-1 most recent pre-conv rows up to the bonus
    // token (raw rows a+1 .. a+W-1), this head's channels, bitwise copies
    {
        __nv_bfloat16 *tail_w = reinterpret_cast<__nv_bfloat16 *>(p.tail);
        for (int idx = tid; idx < (W - 1) * 3 * RP; idx += D) {
            int m = idx / (3 * RP), rem = idx % (3 * RP), part = rem / RP, c = rem % RP;
            uint4 v = *reinterpret_cast<const uint4 *>(&sRaw[(a + 1 + m) * LDR + part * D + c * 8]);
            size_t choff = (size_t)part * H * D + (size_t)h * D + c * 8;
            *reinterpret_cast<uint4 *>(tail_w + ((size_t)r * (W - 1) + m) * Cq + choff) = v;
        }
    }

    // ---------------------------------------------------------------- conv, gates
    // thread c owns channel c of this head's q, k and v
    const int c = tid;
    float xq[VT], xk[VT], xv[VT];
    {
        float wq[4], wk[4], wv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            wq[j] = (j < W) ? p.conv_w[((size_t)h * D + c) * W + j] : 0.f;
            wk[j] = (j < W) ? p.conv_w[((size_t)H * D + h * D + c) * W + j] : 0.f;
            wv[j] = (j < W) ? p.conv_w[((size_t)2 * H * D + h * D + c) * W + j] : 0.f;
        }
#pragma unroll
        for (int t = 0; t < VT; ++t) {
            float yq = 0.f, yk = 0.f, yv = 0.f;
            if (t < ntok) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (j < W) {
                        const __nv_bfloat16 *row = sRaw + (t + j) * LDR;
                        yq = fmaf(wq[j], __bfloat162float(row[c]), yq);
                        yk = fmaf(wk[j], __bfloat162float(row[D + c]), yk);
                        yv = fmaf(wv[j], __bfloat162float(row[2 * D + c]), yv);
                    }
                }
                if (p.conv_act == KDA_CONV_SILU) {
                    yq = yq / (1.f + __expf(-yq));
                    yk = yk / (1.f + __expf(-yk));
                    yv = yv / (1.f + __expf(-yv));
                }
            }
            xq[t] = yq;
            xk[t] = yk;
            xv[t] = yv;
        }
    }
    // decay: x_t = prod_{r<=t} e^{max(-softplus(g_raw), g_min)}, padding e = 1
    float xd[VT];
    {
        float pr = 1.f;
#pragma unroll
        for (int t = 0; t < VT; ++t) {
            if (t < ntok) {
                float graw = __bfloat162float(sGr[t * LDS + c]);
                float sp = fmaxf(graw, 0.f) + log1pf(__expf(-fabsf(graw)));
                pr *= __expf(fmaxf(-sp, p.g_min));
            }
            xd[t] = pr;
        }
        float xa = pr;
#pragma unroll
        for (int t = 0; t < VT; ++t)
            if (t == a) xa = xd[t];
        sXa[c] = xa;
    }
    if (tid < VT) sBeta[tid] = (tid < ntok) ? 1.f / (1.f + __expf(-braw)) : 0.f;

    // input norm: sums of squares over the D channels, per token, for q and k
    {
#pragma unroll
        for (int t = 0; t < VT; ++t) {
            float sq = xq[t] * xq[t], sk = xk[t] * xk[t];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, o);
                sk += __shfl_xor_sync(0xffffffffu, sk, o);
            }
            if (lane == 0) {
                sPart[warp * 32 + t] = sq;
                sPart[NW * 32 + warp * 32 + t] = sk;
            }
        }
    }
    __syncthreads();  // raw rows consumed; partial sums visible
    if (tid < VT) {
        float sq = 0.f, sk = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            sq += sPart[w * 32 + tid];
            sk += sPart[NW * 32 + w * 32 + tid];
        }
        sRq[tid] = rsqrtf(sq + p.eps_in);
        sRk[tid] = rsqrtf(sk + p.eps_in);
    }
    __syncthreads();

    // ---------------------------------------------------------------- operands
    {
        const float xa = sXa[c];
#pragma unroll
        for (int t = 0; t < VT; ++t) {
            float qh = xq[t] * sRq[t], kh = xk[t] * sRk[t];
            float rx = 1.f / xd[t];
            bool live = t < ntok;
            const int e = t * LDS + c;
            split_bf16(live ? qh * xd[t] : 0.f, sQX[e], sQX[PL + e]);
            split_bf16(live ? kh * xd[t] : 0.f, sKX[e], sKX[PL + e]);
            split_bf16(live ? kh * rx : 0.f, sKR[e], sKR[PL + e]);
            split_bf16((t <= a) ? kh * (xa * rx) : 0.f, sKT[e], sKT[PL + e]);
            split_bf16(live ? xv[t] : 0.f, sVv[e], sVv[PL + e]);
        }
    }
    __syncthreads();

    // ---------------------------------------------------------------- A, B (warps 0, 1)
    if (warp < 2) {
        const bool isB = warp == 1;
        const __nv_bfloat16 *lft = isB ? sQX : sKX;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t ah[4], al[4];
            ld_a_rowmajor(ah, lft, LDS, 0, 16 * kk, lane);
            ld_a_rowmajor(al, lft + PL, LDS, 0, 16 * kk, lane);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                int e0 = (8 * nt + gq) * LDS + 16 * kk + 2 * q4;
                uint32_t bh0 = *reinterpret_cast<const uint32_t *>(&sKR[e0]);
                uint32_t bh1 = *reinterpret_cast<const uint32_t *>(&sKR[e0 + 8]);
                uint32_t bl0 = *reinterpret_cast<const uint32_t *>(&sKR[PL + e0]);
                uint32_t bl1 = *reinterpret_cast<const uint32_t *>(&sKR[PL + e0 + 8]);
                mma_bf16(acc[nt], ah, bh0, bh1);
                mma_bf16(acc[nt], ah, bl0, bl1);
                mma_bf16(acc[nt], al, bh0, bh1);
            }
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                int t = gq + 8 * hh, s = 8 * nt + 2 * q4;
                float v0 = acc[nt][2 * hh], v1 = acc[nt][2 * hh + 1];
                if (!isB) {
                    float bt = sBeta[t];
                    sAf[t * 20 + s] = (s < t) ? bt * v0 : 0.f;
                    sAf[t * 20 + s + 1] = (s + 1 < t) ? bt * v1 : 0.f;
                } else {
                    uint32_t hi, lo;
                    split_pack((s <= t) ? v0 : 0.f, (s + 1 <= t) ? v1 : 0.f, hi, lo);
                    *reinterpret_cast<uint32_t *>(&sBm[t * 24 + s]) = hi;
                    *reinterpret_cast<uint32_t *>(&sBm[VT * 24 + t * 24 + s]) = lo;
                }
            }
    }
    __syncthreads();
    // T = (I + A)^{-1}, fp32 forward substitution, one column per lane
    if (warp == 0) {
        const int cc = lane & 15;
        float col[16];
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
            float acc = 0.f;
#pragma unroll
            for (int m = 0; m < rr; ++m) acc = fmaf(sAf[rr * 20 + m], col[m], acc);
            col[rr] = (rr == cc) ? 1.f : ((rr < cc) ? 0.f : -acc);
        }
        if (lane < 16) {
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) sTf[rr * 20 + cc] = col[rr];
        }
    }
    __syncthreads();

    // A fragments of T diag(beta) (hi, lo), shared by W and U~
    uint32_t atb[4], atl[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        int t = gq + 8 * (e & 1), s = 2 * q4 + 8 * (e >> 1);
        split_pack(sTf[t * 20 + s] * sBeta[s], sTf[t * 20 + s + 1] * sBeta[s + 1], atb[e], atl[e]);
    }
    const int cw0 = 32 * warp;  // this warp's 32 columns
    // W = T diag(b) (K . x), columns [cw0, cw0 + 32) of dk
    {
        float acc[4][4];
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[x][e] = 0.f;
#pragma unroll
        for (int np = 0; np < 2; ++np) {
            uint32_t bf[4];
            ld_b_kmajor_rows(bf, sKX, LDS, 0, cw0 + 16 * np, lane);
            mma_bf16(acc[2 * np], atb, bf[0], bf[1]);
            mma_bf16(acc[2 * np + 1], atb, bf[2], bf[3]);
            mma_bf16(acc[2 * np], atl, bf[0], bf[1]);
            mma_bf16(acc[2 * np + 1], atl, bf[2], bf[3]);
        }
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                int t = gq + 8 * hh, col = cw0 + 8 * x + 2 * q4;
                *reinterpret_cast<uint32_t *>(&sW[t * LDS + col]) = pack_bf16(acc[x][2 * hh], acc[x][2 * hh + 1]);
            }
    }
    __syncthreads();

    // [Q x; W] S0 on this warp's value columns
    float aq[4][4], aw[4][4];
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int e = 0; e < 4; ++e) aq[x][e] = aw[x][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        uint32_t fq[4], fw[4];
        ld_a_rowmajor(fq, sQX, LDS, 0, 16 * kk, lane);
        ld_a_rowmajor(fw, sW, LDS, 0, 16 * kk, lane);
#pragma unroll
        for (int np = 0; np < 2; ++np) {
            uint32_t bf[4];
            ld_b_kmajor_rows(bf, sS, LDS, 16 * kk, cw0 + 16 * np, lane);
            mma_bf16(aq[2 * np], fq, bf[0], bf[1]);
            mma_bf16(aq[2 * np + 1], fq, bf[2], bf[3]);
            mma_bf16(aw[2 * np], fw, bf[0], bf[1]);
            mma_bf16(aw[2 * np + 1], fw, bf[2], bf[3]);
        }
    }
    // U = T diag(b) V - W S0
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int e = 0; e < 4; ++e) aw[x][e] = -aw[x][e];
#pragma unroll
    for (int np = 0; np < 2; ++np) {
        uint32_t bf[4];
        uint32_t bl[4];
        ld_b_kmajor_rows(bf, sVv, LDS, 0, cw0 + 16 * np, lane);
        ld_b_kmajor_rows(bl, sVv + PL, LDS, 0, cw0 + 16 * np, lane);
        mma_bf16(aw[2 * np], atb, bf[0], bf[1]);
        mma_bf16(aw[2 * np + 1], atb, bf[2], bf[3]);
        mma_bf16(aw[2 * np], atb, bl[0], bl[1]);
        mma_bf16(aw[2 * np + 1], atb, bl[2], bl[3]);
        mma_bf16(aw[2 * np], atl, bf[0], bf[1]);
        mma_bf16(aw[2 * np + 1], atl, bf[2], bf[3]);
    }
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            int t = gq + 8 * hh, col = cw0 + 8 * x + 2 * q4;
            uint32_t hi, lo;
            split_pack(aw[x][2 * hh], aw[x][2 * hh + 1], hi, lo);
            *reinterpret_cast<uint32_t *>(&sU[t * LDS + col]) = hi;
            *reinterpret_cast<uint32_t *>(&sU[PL + t * LDS + col]) = lo;
        }
    __syncwarp();
    // O = scale (Q x S0 + B U)
    {
        uint32_t fb[4], fbl[4];
        ld_a_rowmajor(fb, sBm, 24, 0, 0, lane);
        ld_a_rowmajor(fbl, sBm + VT * 24, 24, 0, 0, lane);
#pragma unroll
        for (int np = 0; np < 2; ++np) {
            uint32_t bf[4], bl[4];
            ld_b_kmajor_rows(bf, sU, LDS, 0, cw0 + 16 * np, lane);
            ld_b_kmajor_rows(bl, sU + PL, LDS, 0, cw0 + 16 * np, lane);
            mma_bf16(aq[2 * np], fb, bf[0], bf[1]);
            mma_bf16(aq[2 * np + 1], fb, bf[2], bf[3]);
            mma_bf16(aq[2 * np], fb, bl[0], bl[1]);
            mma_bf16(aq[2 * np + 1], fb, bl[2], bl[3]);
            mma_bf16(aq[2 * np], fbl, bf[0], bf[1]);
            mma_bf16(aq[2 * np + 1], fbl, bf[2], bf[3]);
        }
    }
    float ss[2] = {0.f, 0.f};
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            aq[x][e] *= p.scale;
            ss[e >> 1] += aq[x][e] * aq[x][e];
        }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        ss[hh] += __shfl_xor_sync(0xffffffffu, ss[hh], 1);
        ss[hh] += __shfl_xor_sync(0xffffffffu, ss[hh], 2);
    }
    if (q4 == 0) {
        sPart[warp * 32 + gq] = ss[0];
        sPart[warp * 32 + gq + 8] = ss[1];
    }
    __syncthreads();  // also: every warp is done reading S0 as an MMA operand
    {
        __nv_bfloat16 *og = reinterpret_cast<__nv_bfloat16 *>(p.o);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            int t = gq + 8 * hh;
            float tot = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) tot += sPart[w * 32 + t];
            float rs = rsqrtf(tot / D + p.eps_out);
            if (t >= a && t < ntok) {
                size_t orow = (((size_t)r * (Wd + 1) + (t - a)) * H + h) * D;
#pragma unroll
                for (int x = 0; x < 4; ++x) {
                    int col = cw0 + 8 * x + 2 * q4;
                    float v0 = aq[x][2 * hh] * rs * p.out_w[col];
                    float v1 = aq[x][2 * hh + 1] * rs * p.out_w[col + 1];
                    *reinterpret_cast<uint32_t *>(og + orow + col) = pack_bf16(v0, v1);
                }
            }
        }
    }

    // ---------------------------------------------------------------- state after the bonus token
    //   S_a = Diag(x_a) S0 + K~^T U, rows in blocks of 16, this warp's columns
#pragma unroll 1
    for (int mb = 0; mb < D / 16; ++mb) {
        float acc[4][4];
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                int row = 16 * mb + gq + 8 * hh, col = cw0 + 8 * x + 2 * q4;
                float2 s0 = unpack_bf16(*reinterpret_cast<const uint32_t *>(&sS[row * LDS + col]));
                float xa = sXa[row];
                acc[x][2 * hh] = xa * s0.x;
                acc[x][2 * hh + 1] = xa * s0.y;
            }
        uint32_t ak[4], akl[4];
        ld_a_transposed(ak, sKT, LDS, 16 * mb, 0, lane);
        ld_a_transposed(akl, sKT + PL, LDS, 16 * mb, 0, lane);
#pragma unroll
        for (int np = 0; np < 2; ++np) {
            uint32_t bf[4], bl[4];
            ld_b_kmajor_rows(bf, sU, LDS, 0, cw0 + 16 * np, lane);
            ld_b_kmajor_rows(bl, sU + PL, LDS, 0, cw0 + 16 * np, lane);
            mma_bf16(acc[2 * np], ak, bf[0], bf[1]);
            mma_bf16(acc[2 * np + 1], ak, bf[2], bf[3]);
            mma_bf16(acc[2 * np], ak, bl[0], bl[1]);
            mma_bf16(acc[2 * np + 1], ak, bl[2], bl[3]);
            mma_bf16(acc[2 * np], akl, bf[0], bf[1]);
            mma_bf16(acc[2 * np + 1], akl, bf[2], bf[3]);
        }
#pragma unroll
        for (int x = 0; x < 4; ++x)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                int row = 16 * mb + gq + 8 * hh, col = cw0 + 8 * x + 2 * q4;
                *reinterpret_cast<uint32_t *>(&sS[row * LDS + col]) = pack_bf16(acc[x][2 * hh], acc[x][2 * hh + 1]);
            }
    }
    __syncthreads();
    for (int idx = tid; idx < D * RP; idx += D) {
        int row = idx / RP, cc = idx % RP;
        *reinterpret_cast<uint4 *>(stg + (size_t)row * D + cc * 8) =
            *reinterpret_cast<const uint4 *>(&sS[row * LDS + cc * 8]);
    }
}

template <int D>
static cudaError_t launch_verify_t(const VerifyArgs &a, cudaStream_t st) {
    using L = VerifySmem<D>;
    auto kern = kda_verify_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::bytes);
    if (e != cudaSuccess) return e;
    size_t blocks = (size_t)a.R * a.H;
    kern<<<(unsigned)blocks, D, L::bytes, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_verify(const VerifyArgs &a, cudaStream_t st) {
    if (a.R <= 0) return cudaSuccess;
    // by shape: one token per request (no draft window) takes the one-step
    // kernel, d = 128 the tensor-memory kernel, d = 64 the warp-level kernel
    if (a.Wd == 0) return launch_decode_token(a, st);
    if (a.dk == 128 && a.dv == 128) return launch_verify_tc(a, st);
    if (a.dk == 64 && a.dv == 64) return launch_verify_t<64>(a, st);
    return cudaErrorInvalidValue;
}

}  // namespace kda
