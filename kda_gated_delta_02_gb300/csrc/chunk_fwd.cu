// chunk_fwd.cu -- chunkwise KDA prefill on sm_103a.
//
// One CTA (16 warps) walks one (segment, head, dv-tile) unit chunk by chunk,
// 64 tokens per chunk ("Noyaux KDA et FlashKDA", section "FlashKDA : le noyau
// par blocs": parallel within a chunk, serial between chunks).  The fp32
// state tile lives in registers for the whole walk; every product inside a
// chunk runs on the tensor cores with fp32 accumulation, and the dependency
// inverse is fp32 throughout ("Dentro de los esfuerzos de optimizacion de
// Kimi K3", "Nota tecnica: Precision del KDA y memoria on-chip").
//
// Chunk algebra (gamma_t = sum_{r<=t} max(g_r, g_min), per key channel):
//   A[t,s] = b_t sum_c k_tc k_sc e^{gamma_tc - gamma_sc}   (s < t)
//   B[t,s] =     sum_c q_tc k_sc e^{gamma_tc - gamma_sc}   (s <= t)
//   T = (I + A)^{-1};  W = T diag(b)(K . e^gamma);  U~ = T diag(b) V
//   U = U~ - W S;  O = scale ((Q . e^gamma) S + B U)
//   S <- Diag(e^{gamma_63}) S + (K . e^{gamma_63 - gamma})^T U
//
// Dense causal tiles ("Noyaux KDA et FlashKDA", "Le role de la decroissance
// bornee"): the chunk is cut into four 16-token blocks; with b_i the token
// just before block i, every factor e^{gamma_t - gamma_s} is written as
//   x_t * (1/x_s)                         (s, t in the same block i)
//   x_t * c_ij * y_s                      (s in block j < i)
// with x_t = e^{gamma_t - gamma_{b_i}}, y_s = e^{gamma_{b_{j+1}} - gamma_s}
// (both in [e^{-80}, 1] because g >= -5 and a block holds 16 tokens) and a
// per-channel block factor c_ij <= 1.  1/x_s <= e^{80} < FLT_MAX, so each
// causal tile is one dense bf16 product with no overflow; where a factor <= 1
// underflows, the true product is itself below FLT_MIN.  x and y come from
// running products of e^{g} inside each block (one exp per input element).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

constexpr int CH = 64;         // chunk length
constexpr int NTHR = 512;      // 16 warps
constexpr int NWARP = NTHR / 32;

// per-channel vector rows in shared memory
constexpr int V_GB = 0;      // 0..4 : e^{gamma_{b_i}}, i = 0..4 (4 = chunk end)
constexpr int V_C = 5;       // 5..10: c_ij, (1,0) (2,0) (2,1) (3,0) (3,1) (3,2)
constexpr int V_CC = 11;     // 11..14: e^{gamma_63 - gamma_{b_{i+1}}}
constexpr int V_RD = 15;     // 15..18: block decays delta_i, then 1/delta_i
constexpr int NVEC = 20;

__device__ __forceinline__ int vrow_right(int i, int j) {
    return (j == i) ? (V_RD + i) : (V_C + (i * (i - 1)) / 2 + j);
}

template <int DK, int DVT>
struct ChunkSmem {
    static constexpr int LDB = DK + 8;   // bf16 [64][DK] rows
    static constexpr int LDF = DK + 8;   // fp32 [64][DK] rows
    static constexpr int LDV = DVT + 8;  // bf16 [..][DVT] rows
    static constexpr int LDA = 72;       // fp32 / bf16 [64][64] rows
    static constexpr int off_q = 0;
    static constexpr int off_k = off_q + CH * LDB * 2;
    static constexpr int off_v = off_k + CH * LDB * 2;
    static constexpr int off_x = off_v + CH * LDV * 2;
    static constexpr int off_y = off_x + CH * LDF * 4;
    static constexpr int off_beta = off_y + CH * LDF * 4;
    static constexpr int off_a = off_beta + CH * 4;
    static constexpr int off_t = off_a + CH * LDA * 4;
    static constexpr int off_bm = off_t + CH * LDA * 4;
    static constexpr int off_s = off_bm + CH * LDA * 2;
    static constexpr int off_vec = off_s + DK * LDV * 2;
    static constexpr int bytes = off_vec + NVEC * DK * 4;
    static_assert(CH * LDV * 2 <= CH * LDA * 4, "U tile must fit in the A buffer");
};

template <int DK, int DVT, bool IN_BF16>
__global__ void __launch_bounds__(NTHR, 1) kda_chunk_kernel(ChunkArgs p) {
    using L = ChunkSmem<DK, DVT>;
    using in_t = typename std::conditional<IN_BF16, __nv_bfloat16, float>::type;
    constexpr int LDB = L::LDB, LDF = L::LDF, LDV = L::LDV, LDA = L::LDA;
    constexpr int MB = DK / 16;         // row blocks of the state tile
    constexpr int NSPLIT = NWARP / MB;  // column splits of the state tile
    constexpr int CPW = DVT / NSPLIT;   // state columns per warp
    constexpr int NT8 = CPW / 8;
    constexpr int NT1 = DVT / 16;       // n8 tiles per warp in [Q~;W] S (half of DVT)
    constexpr int NTW = DK / 16;        // n8 tiles per warp in W (half of DK)
    static_assert(NT8 % 2 == 0 && NT1 % 2 == 0 && NTW % 2 == 0, "x4 fragment loads");

    extern __shared__ __align__(128) unsigned char smem[];
    __nv_bfloat16 *sQ = reinterpret_cast<__nv_bfloat16 *>(smem + L::off_q);
    __nv_bfloat16 *sK = reinterpret_cast<__nv_bfloat16 *>(smem + L::off_k);   // -> K.e^gamma
    __nv_bfloat16 *sV = reinterpret_cast<__nv_bfloat16 *>(smem + L::off_v);
    float *sX = reinterpret_cast<float *>(smem + L::off_x);                    // g -> x
    float *sY = reinterpret_cast<float *>(smem + L::off_y);                    // y
    __nv_bfloat16 *sKt = reinterpret_cast<__nv_bfloat16 *>(smem + L::off_y);  // K~ (after y)
    __nv_bfloat16 *sW = sKt + CH * LDB;                                        // W  (after y)
    float *sBeta = reinterpret_cast<float *>(smem + L::off_beta);
    float *sA = reinterpret_cast<float *>(smem + L::off_a);
    __nv_bfloat16 *sU = reinterpret_cast<__nv_bfloat16 *>(smem + L::off_a);  // U (after A)
    float *sT = reinterpret_cast<float *>(smem + L::off_t);
    __nv_bfloat16 *sBm = reinterpret_cast<__nv_bfloat16 *>(smem + L::off_bm);
    __nv_bfloat16 *sS = reinterpret_cast<__nv_bfloat16 *>(smem + L::off_s);
    float *sVec = reinterpret_cast<float *>(smem + L::off_vec);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, q4 = lane & 3;
    const int unit = blockIdx.x, h = blockIdx.y, tile = blockIdx.z;
    const int H = p.H;

    // ---------------------------------------------------------------- work unit
    int n, t0, t1;
    bool last_seg = true;
    if (p.mode == MODE_SEQ) {
        n = unit;
        t0 = p.cu_seqlens[n];
        t1 = p.cu_seqlens[n + 1];
        if (t0 < 0 || t1 < t0 || t1 > p.T) {
            if (tid == 0) report_status(p.status, KDA_STATUS_BAD_SEQLENS);
            return;
        }
    } else if (p.seg_table) {
        if (unit >= *p.seg_count) return;
        const int4 e = reinterpret_cast<const int4 *>(p.seg_table)[unit];
        n = e.x;
        t0 = e.y;
        t1 = e.z;
        last_seg = e.w != 0;
    } else {  // one sequence cut into fixed-length segments
        n = 0;
        t0 = unit * p.seg_len;
        t1 = min(p.T, t0 + p.seg_len);
        last_seg = t1 == p.T;
    }
    // start of this unit's sequence (checkpoint positions are relative to it)
    const int seq0 = (p.mode == MODE_SEQ) ? t0 : ((p.seg_table && p.cu_seqlens) ? p.cu_seqlens[n] : 0);
    // columns: in transition mode the tile walks the augmented state [M | N]
    const int colbase = tile * DVT;
    bool m_part = false;
    int vcol0 = colbase;
    if (p.mode == MODE_TRANSITION) {
        m_part = colbase < DK;
        vcol0 = m_part ? 0 : colbase - DK;
    }
    const bool has_v = !m_part;
    const bool need_q = p.mode != MODE_TRANSITION;  // transitions produce no output
    const int dv = p.dv;

    // ---------------------------------------------------------------- state init
    const int mb = warp % MB, cs = warp / MB;
    float sreg[NT8][4];
#pragma unroll
    for (int nt = 0; nt < NT8; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            int row = 16 * mb + gq + 8 * (e >> 1);
            int col = cs * CPW + 8 * nt + 2 * q4 + (e & 1);
            float v0 = 0.f;
            if (p.mode == MODE_TRANSITION) {
                v0 = (m_part && row == colbase + col) ? 1.f : 0.f;
            } else {
                const float *src = (p.mode == MODE_SEQ) ? p.S_init : p.S_in;
                if (src) {
                    size_t sidx = (p.mode == MODE_SEQ) ? (size_t)n : (size_t)unit;
                    v0 = src[((sidx * H + h) * DK + row) * (size_t)dv + vcol0 + col];
                }
            }
            sreg[nt][e] = v0;
        }
    auto store_state_bf16 = [&]() {
#pragma unroll
        for (int nt = 0; nt < NT8; ++nt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                int row = 16 * mb + gq + 8 * hh;
                int col = cs * CPW + 8 * nt + 2 * q4;
                *reinterpret_cast<uint32_t *>(&sS[row * LDV + col]) =
                    pack_bf16(sreg[nt][2 * hh], sreg[nt][2 * hh + 1]);
            }
    };
    store_state_bf16();

    const float g_min = p.g_min;
    const float scale = p.scale;
    const in_t *qg = reinterpret_cast<const in_t *>(p.q);
    const in_t *kg = reinterpret_cast<const in_t *>(p.k);
    const in_t *vg = reinterpret_cast<const in_t *>(p.v);

    for (int tc = t0; tc < t1; tc += CH) {
        const int Lc = min(CH, t1 - tc);
        // ------------------------------------------------------------ loads
        if constexpr (IN_BF16) {
            constexpr int QCH = DK / 8;  // 16-byte pieces per row
            for (int idx = tid; idx < CH * QCH; idx += NTHR) {
                int r = idx / QCH, c = idx % QCH;
                bool ok = r < Lc;
                size_t row = ok ? ((size_t)(tc + r) * H + h) : 0;
                if (need_q) cp_async16(&sQ[r * LDB + c * 8], qg + row * DK + c * 8, ok);
                cp_async16(&sK[r * LDB + c * 8], kg + row * DK + c * 8, ok);
            }
            constexpr int VCH = DVT / 8;
            for (int idx = tid; idx < CH * VCH; idx += NTHR) {
                int r = idx / VCH, c = idx % VCH;
                bool ok = r < Lc && has_v;
                size_t row = ok ? ((size_t)(tc + r) * H + h) : 0;
                cp_async16(&sV[r * LDV + c * 8], vg + row * dv + (ok ? vcol0 : 0) + c * 8, ok);
            }
        } else {
            constexpr int Q4 = DK / 4;
            for (int idx = tid; idx < CH * Q4; idx += NTHR) {
                int r = idx / Q4, c = idx % Q4;
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
                if (r < Lc) {
                    size_t row = (size_t)(tc + r) * H + h;
                    if (need_q) a = *reinterpret_cast<const float4 *>(qg + row * DK + c * 4);
                    b = *reinterpret_cast<const float4 *>(kg + row * DK + c * 4);
                }
                uint2 pa = make_uint2(pack_bf16(a.x, a.y), pack_bf16(a.z, a.w));
                uint2 pb = make_uint2(pack_bf16(b.x, b.y), pack_bf16(b.z, b.w));
                *reinterpret_cast<uint2 *>(&sQ[r * LDB + c * 4]) = pa;
                *reinterpret_cast<uint2 *>(&sK[r * LDB + c * 4]) = pb;
            }
            constexpr int V4 = DVT / 4;
            for (int idx = tid; idx < CH * V4; idx += NTHR) {
                int r = idx / V4, c = idx % V4;
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
                if (r < Lc && has_v) {
                    size_t row = (size_t)(tc + r) * H + h;
                    a = *reinterpret_cast<const float4 *>(vg + row * dv + vcol0 + c * 4);
                }
                *reinterpret_cast<uint2 *>(&sV[r * LDV + c * 4]) =
                    make_uint2(pack_bf16(a.x, a.y), pack_bf16(a.z, a.w));
            }
        }
        {
            constexpr int GCH = DK / 4;
            for (int idx = tid; idx < CH * GCH; idx += NTHR) {
                int r = idx / GCH, c = idx % GCH;
                bool ok = r < Lc;
                size_t row = ok ? ((size_t)(tc + r) * H + h) : 0;
                cp_async16(&sX[r * LDF + c * 4], p.g + row * DK + c * 4, ok);
            }
            if (tid < CH) {
                bool ok = tid < Lc;
                size_t row = ok ? ((size_t)(tc + tid) * H + h) : 0;
                cp_async4(&sBeta[tid], p.beta + row, ok);
            }
        }
        cp_async_commit();
        cp_async_wait_all();
        __syncthreads();

        // ------------------------------------------------------------ decay scan
        for (int task = tid; task < 4 * DK; task += NTHR) {
            int ch = task % DK, blk = task / DK;
            float e[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) e[r] = __expf(fmaxf(sX[(16 * blk + r) * LDF + ch], g_min));
            float pr = 1.f;
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                pr *= e[r];
                sX[(16 * blk + r) * LDF + ch] = pr;
            }
            float sf = 1.f;
#pragma unroll
            for (int r = 15; r >= 0; --r) {
                sY[(16 * blk + r) * LDF + ch] = sf;
                sf *= e[r];
            }
            sVec[(V_RD + blk) * DK + ch] = pr;
        }
        __syncthreads();
        if (tid < DK) {
            const int ch = tid;
            float d0 = sVec[(V_RD + 0) * DK + ch], d1 = sVec[(V_RD + 1) * DK + ch];
            float d2 = sVec[(V_RD + 2) * DK + ch], d3 = sVec[(V_RD + 3) * DK + ch];
            sVec[(V_GB + 0) * DK + ch] = 1.f;
            sVec[(V_GB + 1) * DK + ch] = d0;
            sVec[(V_GB + 2) * DK + ch] = d0 * d1;
            sVec[(V_GB + 3) * DK + ch] = (d0 * d1) * d2;
            sVec[(V_GB + 4) * DK + ch] = ((d0 * d1) * d2) * d3;
            sVec[(V_C + 0) * DK + ch] = 1.f;      // c10
            sVec[(V_C + 1) * DK + ch] = d1;       // c20
            sVec[(V_C + 2) * DK + ch] = 1.f;      // c21
            sVec[(V_C + 3) * DK + ch] = d1 * d2;  // c30
            sVec[(V_C + 4) * DK + ch] = d2;       // c31
            sVec[(V_C + 5) * DK + ch] = 1.f;      // c32
            sVec[(V_CC + 0) * DK + ch] = (d1 * d2) * d3;
            sVec[(V_CC + 1) * DK + ch] = d2 * d3;
            sVec[(V_CC + 2) * DK + ch] = d3;
            sVec[(V_CC + 3) * DK + ch] = 1.f;
            sVec[(V_RD + 0) * DK + ch] = 1.f / d0;
            sVec[(V_RD + 1) * DK + ch] = 1.f / d1;
            sVec[(V_RD + 2) * DK + ch] = 1.f / d2;
            sVec[(V_RD + 3) * DK + ch] = 1.f / d3;
        }
        __syncthreads();

        // ------------------------------------------------------------ A and B tiles
        {
            const int i = warp >> 2;           // row block
            const int isB = (warp >> 1) & 1;   // 0: A (keys), 1: B (queries)
            const int hf = warp & 1;           // half of the column tiles
            const __nv_bfloat16 *lsrc = isB ? sQ : sK;
            if (isB && !need_q) goto ab_done;
            float acc[4][4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[a][e] = 0.f;
#pragma unroll
            for (int kk = 0; kk < DK / 16; ++kk) {
                uint32_t af[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int t = 16 * i + gq + 8 * (e & 1);
                    int ch = 16 * kk + 2 * q4 + 8 * (e >> 1);
                    float2 kv = unpack_bf16(*reinterpret_cast<const uint32_t *>(&lsrc[t * LDB + ch]));
                    float2 xv = *reinterpret_cast<const float2 *>(&sX[t * LDF + ch]);
                    af[e] = pack_bf16(kv.x * xv.x, kv.y * xv.y);
                }
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    if (a <= i) {
                        int nt = hf * (i + 1) + a;
                        int s = 8 * nt + gq;
                        int j = nt >> 1;
                        const float *vr = sVec + vrow_right(i, j) * DK;
                        uint32_t bf[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            int ch = 16 * kk + 2 * q4 + 8 * e;
                            float2 kv = unpack_bf16(*reinterpret_cast<const uint32_t *>(&sK[s * LDB + ch]));
                            float2 yv = *reinterpret_cast<const float2 *>(&sY[s * LDF + ch]);
                            float2 fv = *reinterpret_cast<const float2 *>(&vr[ch]);
                            bf[e] = pack_bf16(kv.x * (yv.x * fv.x), kv.y * (yv.y * fv.y));
                        }
                        mma_bf16(acc[a], af, bf[0], bf[1]);
                    }
                }
            }
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                if (a <= i) {
                    int nt = hf * (i + 1) + a;
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        int t = 16 * i + gq + 8 * hh;
                        int s = 8 * nt + 2 * q4;
                        float v0 = acc[a][2 * hh], v1 = acc[a][2 * hh + 1];
                        if (!isB) {
                            float bt = sBeta[t];
                            float2 w;
                            w.x = (s < t) ? bt * v0 : 0.f;
                            w.y = (s + 1 < t) ? bt * v1 : 0.f;
                            *reinterpret_cast<float2 *>(&sA[t * LDA + s]) = w;
                        } else {
                            *reinterpret_cast<uint32_t *>(&sBm[t * LDA + s]) =
                                pack_bf16((s <= t) ? v0 : 0.f, (s + 1 <= t) ? v1 : 0.f);
                        }
                    }
                }
            }
        }
    ab_done:
        __syncthreads();

        // ------------------------------------------------------------ inverse (diagonal blocks)
        //   warps 0-3: T_ii = (I + A_ii)^{-1} by forward substitution, fp32
        //   warps 4-15: K . e^gamma (in place of K) and K~ (in place of y)
        if (warp < 4) {
            const int i = warp, c = lane & 15;
            float col[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float acc = 0.f;
#pragma unroll
                for (int m = 0; m < r; ++m) acc = fmaf(sA[(16 * i + r) * LDA + 16 * i + m], col[m], acc);
                col[r] = (r == c) ? 1.f : ((r < c) ? 0.f : -acc);
            }
            if (lane < 16) {
#pragma unroll
                for (int r = 0; r < 16; ++r) sT[(16 * i + r) * LDA + 16 * i + c] = col[r];
            }
        } else {
            constexpr int NPAIR = CH * DK / 2;
            constexpr int PER = (NPAIR + (NTHR - 128) - 1) / (NTHR - 128);
            uint32_t kt[PER];
            const int base = tid - 128;
#pragma unroll
            for (int u = 0; u < PER; ++u) {
                int pidx = base + u * (NTHR - 128);
                kt[u] = 0;
                if (pidx < NPAIR) {
                    int t = pidx / (DK / 2), ch = 2 * (pidx % (DK / 2));
                    int blk = t >> 4;
                    float2 kv = unpack_bf16(*reinterpret_cast<const uint32_t *>(&sK[t * LDB + ch]));
                    float2 xv = *reinterpret_cast<const float2 *>(&sX[t * LDF + ch]);
                    float2 yv = *reinterpret_cast<const float2 *>(&sY[t * LDF + ch]);
                    float2 gb = *reinterpret_cast<const float2 *>(&sVec[(V_GB + blk) * DK + ch]);
                    float2 cc = *reinterpret_cast<const float2 *>(&sVec[(V_CC + blk) * DK + ch]);
                    *reinterpret_cast<uint32_t *>(&sK[t * LDB + ch]) =
                        pack_bf16(kv.x * (xv.x * gb.x), kv.y * (xv.y * gb.y));
                    kt[u] = pack_bf16(kv.x * (yv.x * cc.x), kv.y * (yv.y * cc.y));
                }
            }
            asm volatile("bar.sync 1, %0;\n" ::"n"(NTHR - 128));
#pragma unroll
            for (int u = 0; u < PER; ++u) {
                int pidx = base + u * (NTHR - 128);
                if (pidx < NPAIR) {
                    int t = pidx / (DK / 2), ch = 2 * (pidx % (DK / 2));
                    *reinterpret_cast<uint32_t *>(&sKt[t * LDB + ch]) = kt[u];
                }
            }
        }
        __syncthreads();

        // ------------------------------------------------------------ inverse (off-diagonal)
        // T_ij = -T_ii sum_{m=j}^{i-1} A_im T_mj, by distance d = i - j
#pragma unroll 1
        for (int d = 1; d < 4; ++d) {
            const int nel = (4 - d) * 256;
            float xv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                int e = tid + u * NTHR;
                xv[u] = 0.f;
                if (e < nel) {
                    int b = e >> 8, r = (e >> 4) & 15, c = e & 15;
                    int i = b + d, j = b;
                    float acc = 0.f;
                    for (int m = 16 * j; m < 16 * i; ++m)
                        acc = fmaf(sA[(16 * i + r) * LDA + m], sT[m * LDA + 16 * j + c], acc);
                    xv[u] = acc;
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                int e = tid + u * NTHR;
                if (e < nel) {
                    int b = e >> 8, r = (e >> 4) & 15, c = e & 15;
                    sT[(16 * (b + d) + r) * LDA + 16 * b + c] = xv[u];
                }
            }
            __syncthreads();
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                int e = tid + u * NTHR;
                if (e < nel) {
                    int b = e >> 8, r = (e >> 4) & 15, c = e & 15;
                    int i = b + d, j = b;
                    float acc = 0.f;
                    for (int m = 0; m <= r; ++m)
                        acc = fmaf(sT[(16 * i + r) * LDA + 16 * i + m], sT[(16 * i + m) * LDA + 16 * j + c], acc);
                    xv[u] = -acc;
                }
            }
            __syncthreads();
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                int e = tid + u * NTHR;
                if (e < nel) {
                    int b = e >> 8, r = (e >> 4) & 15, c = e & 15;
                    sT[(16 * (b + d) + r) * LDA + 16 * b + c] = xv[u];
                }
            }
            __syncthreads();
        }

        // ------------------------------------------------------------ W (to smem)
        const int rb = warp & 7, hf = warp >> 3;
        if (rb < 4) {
            const int i = rb, chh = hf;
            float acc[NTW][4];
#pragma unroll
            for (int a = 0; a < NTW; ++a)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[a][e] = 0.f;
            for (int m = 0; m <= i; ++m) {
                uint32_t af[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int t = 16 * i + gq + 8 * (e & 1);
                    int s = 16 * m + 2 * q4 + 8 * (e >> 1);
                    float2 tv = *reinterpret_cast<const float2 *>(&sT[t * LDA + s]);
                    af[e] = pack_bf16(tv.x * sBeta[s], tv.y * sBeta[s + 1]);
                }
#pragma unroll
                for (int np = 0; np < NTW / 2; ++np) {
                    uint32_t bf[4];
                    ld_b_kmajor_rows(bf, sK, LDB, 16 * m, chh * (DK / 2) + 16 * np, lane);
                    mma_bf16(acc[2 * np], af, bf[0], bf[1]);
                    mma_bf16(acc[2 * np + 1], af, bf[2], bf[3]);
                }
            }
#pragma unroll
            for (int a = 0; a < NTW; ++a)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    int t = 16 * i + gq + 8 * hh;
                    int ch = chh * (DK / 2) + 8 * a + 2 * q4;
                    *reinterpret_cast<uint32_t *>(&sW[t * LDB + ch]) =
                        pack_bf16(acc[a][2 * hh], acc[a][2 * hh + 1]);
                }
        }
        __syncthreads();

        // ------------------------------------------------------------ [Q~; W] S
        float acc1[NT1][4];
#pragma unroll
        for (int a = 0; a < NT1; ++a)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc1[a][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < DK / 16; ++kk) {
            uint32_t af[4];
            if (rb < 4 && !need_q) break;
            if (rb < 4) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int t = 16 * rb + gq + 8 * (e & 1);
                    int ch = 16 * kk + 2 * q4 + 8 * (e >> 1);
                    float2 qv = unpack_bf16(*reinterpret_cast<const uint32_t *>(&sQ[t * LDB + ch]));
                    float2 xv = *reinterpret_cast<const float2 *>(&sX[t * LDF + ch]);
                    float2 gb = *reinterpret_cast<const float2 *>(&sVec[(V_GB + rb) * DK + ch]);
                    af[e] = pack_bf16(qv.x * (xv.x * gb.x), qv.y * (xv.y * gb.y));
                }
            } else {
                ld_a_rowmajor(af, sW, LDB, 16 * (rb - 4), 16 * kk, lane);
            }
#pragma unroll
            for (int np = 0; np < NT1 / 2; ++np) {
                uint32_t bf[4];
                ld_b_kmajor_rows(bf, sS, LDV, 16 * kk, hf * (DVT / 2) + 16 * np, lane);
                mma_bf16(acc1[2 * np], af, bf[0], bf[1]);
                mma_bf16(acc1[2 * np + 1], af, bf[2], bf[3]);
            }
        }
        // W rows: U = U~ - W S, with U~ = T diag(b) V accumulated onto -WS
        if (rb >= 4) {
            const int i = rb - 4;
#pragma unroll
            for (int a = 0; a < NT1; ++a)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc1[a][e] = -acc1[a][e];
            for (int m = 0; m <= i; ++m) {
                uint32_t af[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int t = 16 * i + gq + 8 * (e & 1);
                    int s = 16 * m + 2 * q4 + 8 * (e >> 1);
                    float2 tv = *reinterpret_cast<const float2 *>(&sT[t * LDA + s]);
                    af[e] = pack_bf16(tv.x * sBeta[s], tv.y * sBeta[s + 1]);
                }
#pragma unroll
                for (int np = 0; np < NT1 / 2; ++np) {
                    uint32_t bf[4];
                    ld_b_kmajor_rows(bf, sV, LDV, 16 * m, hf * (DVT / 2) + 16 * np, lane);
                    mma_bf16(acc1[2 * np], af, bf[0], bf[1]);
                    mma_bf16(acc1[2 * np + 1], af, bf[2], bf[3]);
                }
            }
        }
        __syncthreads();  // all reads of sA / sT / sS done
        if (rb >= 4) {
            const int i = rb - 4;
#pragma unroll
            for (int a = 0; a < NT1; ++a)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    int t = 16 * i + gq + 8 * hh;
                    int col = hf * (DVT / 2) + 8 * a + 2 * q4;
                    *reinterpret_cast<uint32_t *>(&sU[t * LDV + col]) =
                        pack_bf16(acc1[a][2 * hh], acc1[a][2 * hh + 1]);
                }
        }
        __syncthreads();

        // ------------------------------------------------------------ O = Q~S + B U
        if (rb < 4 && p.mode != MODE_TRANSITION) {
            for (int m = 0; m <= rb; ++m) {
                uint32_t af[4];
                ld_a_rowmajor(af, sBm, LDA, 16 * rb, 16 * m, lane);
#pragma unroll
                for (int np = 0; np < NT1 / 2; ++np) {
                    uint32_t bf[4];
                    ld_b_kmajor_rows(bf, sU, LDV, 16 * m, hf * (DVT / 2) + 16 * np, lane);
                    mma_bf16(acc1[2 * np], af, bf[0], bf[1]);
                    mma_bf16(acc1[2 * np + 1], af, bf[2], bf[3]);
                }
            }
            in_t *og = reinterpret_cast<in_t *>(p.o);
#pragma unroll
            for (int a = 0; a < NT1; ++a)
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    int t = 16 * rb + gq + 8 * hh;
                    if (t < Lc) {
                        int col = vcol0 + hf * (DVT / 2) + 8 * a + 2 * q4;
                        size_t off = ((size_t)(tc + t) * H + h) * dv + col;
                        float v0 = scale * acc1[a][2 * hh], v1 = scale * acc1[a][2 * hh + 1];
                        if constexpr (IN_BF16) {
                            *reinterpret_cast<uint32_t *>(og + off) = pack_bf16(v0, v1);
                        } else {
                            *reinterpret_cast<float2 *>(og + off) = make_float2(v0, v1);
                        }
                    }
                }
        }

        // ------------------------------------------------------------ S update
        {
#pragma unroll
            for (int nt = 0; nt < NT8; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    int row = 16 * mb + gq + 8 * (e >> 1);
                    sreg[nt][e] *= sVec[(V_GB + 4) * DK + row];
                }
#pragma unroll
            for (int kk = 0; kk < CH / 16; ++kk) {
                uint32_t af[4];
                ld_a_transposed(af, sKt, LDB, 16 * mb, 16 * kk, lane);
#pragma unroll
                for (int np = 0; np < NT8 / 2; ++np) {
                    uint32_t bf[4];
                    ld_b_kmajor_rows(bf, sU, LDV, 16 * kk, cs * CPW + 16 * np, lane);
                    mma_bf16(sreg[2 * np], af, bf[0], bf[1]);
                    mma_bf16(sreg[2 * np + 1], af, bf[2], bf[3]);
                }
            }
            store_state_bf16();
        }
        // checkpoint: the state after token (tc + Lc) when that position of the
        // sequence is a multiple of ckpt_every
        if (p.ckpt && p.mode != MODE_TRANSITION) {
            const int rel = tc + Lc - seq0;
            const int kq = rel / p.ckpt_every - 1;
            if (rel % p.ckpt_every == 0 && kq < p.ckpt_count) {
                float *dst = p.ckpt + (((size_t)n * p.ckpt_count + kq) * H + h) * DK * (size_t)dv;
#pragma unroll
                for (int nt = 0; nt < NT8; ++nt)
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        int row = 16 * mb + gq + 8 * hh;
                        int col = cs * CPW + 8 * nt + 2 * q4;
                        *reinterpret_cast<float2 *>(dst + (size_t)row * dv + vcol0 + col) =
                            make_float2(sreg[nt][2 * hh], sreg[nt][2 * hh + 1]);
                    }
            }
        }
        __syncthreads();
    }

    // ---------------------------------------------------------------- state out
    float *dst = nullptr;
    size_t ld_dst = dv, dst_col0 = vcol0;
    if (p.mode == MODE_SEQ) {
        if (p.S_final) dst = p.S_final + ((size_t)n * H + h) * DK * (size_t)dv;
    } else if (p.mode == MODE_REPLAY) {
        if (p.S_final && last_seg) dst = p.S_final + ((size_t)n * H + h) * DK * (size_t)dv;
    } else {
        if (m_part) {
            dst = p.M_out + ((size_t)unit * H + h) * DK * (size_t)DK;
            ld_dst = DK;
            dst_col0 = colbase;
        } else {
            dst = p.N_out + ((size_t)unit * H + h) * DK * (size_t)dv;
        }
    }
    if (dst) {
#pragma unroll
        for (int nt = 0; nt < NT8; ++nt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                int row = 16 * mb + gq + 8 * hh;
                int col = cs * CPW + 8 * nt + 2 * q4;
                *reinterpret_cast<float2 *>(dst + row * ld_dst + dst_col0 + col) =
                    make_float2(sreg[nt][2 * hh], sreg[nt][2 * hh + 1]);
            }
    }
}

// Segment table for the context-parallel path: every sequence is cut into
// ceil(len / seg_len) segments (at least one, so empty sequences still carry
// their state).  Entry = {sequence, t0, t1, is_last}; seq_first[n] = index of
// the first segment of sequence n, seq_first[N] = total.
__global__ void kda_segment_table_kernel(const int32_t *cu_seqlens, int N, int T, int seg_len,
                                         int P_max, int32_t *table, int32_t *seq_first,
                                         int32_t *seg_count, uint32_t *status) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    int P = 0;
    bool bad = false;
    for (int n = 0; n < N; ++n) {
        int a = cu_seqlens[n], b = cu_seqlens[n + 1];
        seq_first[n] = P;
        if (a < 0 || b < a || b > T) {
            bad = true;
            continue;
        }
        int ns = (b - a + seg_len - 1) / seg_len;
        if (ns < 1) ns = 1;
        for (int s = 0; s < ns; ++s) {
            if (P >= P_max) {
                report_status(status, KDA_STATUS_SEGMENT_OVERFLOW);
                for (int m = n + 1; m <= N; ++m) seq_first[m] = P;  // later sequences: no segment
                *seg_count = P;
                return;
            }
            int s0 = a + s * seg_len;
            int s1 = min(b, s0 + seg_len);
            table[4 * P + 0] = n;
            table[4 * P + 1] = s0;
            table[4 * P + 2] = s1;
            table[4 * P + 3] = (s == ns - 1) ? 1 : 0;
            ++P;
        }
    }
    seq_first[N] = P;
    *seg_count = P;
    if (bad) report_status(status, KDA_STATUS_BAD_SEQLENS);
}

template <int DK, int DVT, bool IN_BF16>
static cudaError_t launch_chunk_t(const ChunkArgs &a, int units, int ntiles, cudaStream_t st) {
    using L = ChunkSmem<DK, DVT>;
    auto kern = kda_chunk_kernel<DK, DVT, IN_BF16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::bytes);
    if (e != cudaSuccess) return e;
    dim3 grid(units, a.H, ntiles);
    kern<<<grid, NTHR, L::bytes, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_chunk(const ChunkArgs &a, int units, int dvt, bool in_bf16, cudaStream_t st) {
    const int width = (a.mode == MODE_TRANSITION) ? a.dk + a.dv : a.dv;
    const int ntiles = width / dvt;
    if (units <= 0 || ntiles <= 0) return cudaSuccess;
#define KDA_DISPATCH(DK_, DVT_)                                                               \
    if (a.dk == DK_ && dvt == DVT_)                                                           \
        return in_bf16 ? launch_chunk_t<DK_, DVT_, true>(a, units, ntiles, st)                \
                       : launch_chunk_t<DK_, DVT_, false>(a, units, ntiles, st);
    KDA_DISPATCH(128, 128)
    KDA_DISPATCH(128, 64)
    KDA_DISPATCH(64, 64)
    KDA_DISPATCH(64, 128)
#undef KDA_DISPATCH
    return cudaErrorInvalidValue;
}

cudaError_t launch_segment_table(const int32_t *cu_seqlens, int N, int T, int seg_len, int P_max,
                                 int32_t *table, int32_t *seq_first, int32_t *seg_count,
                                 uint32_t *status, cudaStream_t st) {
    kda_segment_table_kernel<<<1, 32, 0, st>>>(cu_seqlens, N, T, seg_len, P_max, table, seq_first,
                                                seg_count, status);
    return cudaGetLastError();
}

}  // namespace kda
