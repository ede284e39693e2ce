// chunk_fwd_tc.cu -- chunkwise KDA prefill on the sm_103a tensor cores
// (tcgen05.mma, accumulators in tensor memory), dk = dv = 128, bf16 inputs.
//
// One CTA (16 warps) walks one (segment, head) unit, 64 tokens per chunk
// ("Noyaux KDA et FlashKDA", section "FlashKDA : le noyau par blocs").  The
// fp32 state S^T (dv rows x dk) stays on chip for the whole walk: thread
// (lane quadrant q, column group g) owns row 32q + lane, columns 32g .. 32g+31;
// the state itself lives in tensor memory for the whole walk.  Every product of the
// chunk runs as a tcgen05 MMA with M = 128 on operands staged in shared memory
// in the 128-byte swizzled layouts; transposed forms put dv (or dk) on M:
//   A/B tiles  D[t'][s'] = L[t'] . R[s']    (all 128 L rows x the 160 rows of R_0..R_3;
//                                            block i uses its L rows against R_i)
//   W^T        D[i][t]   = (K e^gamma)^T  (T diag b)^T
//   U~^T       D[j][t]   = V^T (T diag b)^T,      then  -= S^T W^T   ->  U^T
//   O^T        D[j][t]   = S^T Q~^T + U^T B^T
//   S update   S^T <- Diag-cols(e^{gamma_63}) S^T (in place), then += U^T K~ by the MMA
// with R_i[s] = k_s y_s c_{i,j(s)} (1/delta_i on the diagonal block) and
// L[t] = k_t x_t or q_t x_t: the per-16-token-block anchoring that the
// g >= -5 floor makes overflow-free ("Noyaux KDA et FlashKDA", "Le role de la
// decroissance bornee"); x, y are running products of e^{g} inside a block.
// The dependency inverse T = (I + A)^{-1} is fp32 throughout ("Dentro de los
// esfuerzos de optimizacion de Kimi K3", "Nota tecnica: Precision del KDA").
#include <cuda.h>  // CUtensorMap (the encoder is reached through the runtime)
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_umma.cuh"

namespace kda {
namespace tc {

constexpr int D = 128;  // dk = dv
constexpr int CH = 64;
constexpr int NT = 512;

// shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_Q = 0;         // raw q bf16 [64][128]
constexpr uint32_t OFF_K = 16384;     // raw k bf16 [64][128]
constexpr uint32_t OFF_G = 32768;     // raw g f32 [64][128]
constexpr uint32_t OFF_V = 65536;     // V, MN-major (s x dv): two 64-wide halves of [64 s][128 B]
constexpr uint32_t OFF_UN = 81920;    // union, 73728 bytes:
constexpr uint32_t UN_L = 0;          //   L (K-major 128 x 128)         steps 2-3
constexpr uint32_t UN_R = 32768;      //   R = [R_0; R_1; R_2; R_3] (K-major 160 rows x 128)  steps 2-3
constexpr uint32_t R_KB = 160 * 128;  //   its K-block stride (two 64-wide K-blocks, 20480 B each)
// rows of R_i start at row 8 i (i+1): 0, 16, 48, 96 (16 (i+1) rows each)
__host__ __device__ constexpr uint32_t r_row(int i) { return 8u * (uint32_t)(i * (i + 1)); }
constexpr uint32_t UN_AF = 34816;     //   A fp32 [64][68]                steps 4-5
constexpr uint32_t UN_TF = 52224;     //   T fp32 [64][68]
constexpr uint32_t UN_ST = 0;         //   S^T bf16 (K-major 128 x 128)   steps 4-8
constexpr uint32_t UN_W = 32768;      //   W (MN-major: 128 k-rows i x 64 t)
constexpr uint32_t UN_UT = 49152;     //   U^T (K-major 128 x 64)         steps 9-10
constexpr uint32_t OFF_KG = 155648;   // K e^gamma, MN-major (s x dk)
constexpr uint32_t OFF_QT = 172032;   // Q e^gamma, K-major 64 x 128
constexpr uint32_t OFF_KT = 188416;   // K e^{gamma_63 - gamma}, MN-major (s x dk)
constexpr uint32_t OFF_TB = 204800;   // T diag(b), K-major 64 x 64
constexpr uint32_t OFF_BM = 212992;   // B, K-major (64 rows t x 64 s)
constexpr uint32_t OFF_BETA = 221184; // f32 [64]
constexpr uint32_t OFF_PART = 221440; // f32 [2][4][128] half-block products
constexpr uint32_t OFF_DEL = 225536;  // f32 [4][128] block decays
constexpr uint32_t OFF_GAM = 227584;  // f32 [128] chunk decay e^{gamma_63}
constexpr uint32_t OFF_BAR = 228096;  // 6 mbarriers: 4 MMA groups, q/k/g loads, v loads
constexpr uint32_t OFF_TMEM = 228144; // tensor-memory base address
constexpr uint32_t SMEM_BYTES = 228160 + 1024;  // + alignment slack
constexpr int LDF = 68;               // fp32 [64][68] row stride

// tensor-memory columns
//   S^T (fp32, the state, resident for the whole walk; the U^T K~ update
//   accumulates onto it) | L R^T (160 columns) | W^T | U^T | O^T
constexpr uint32_t TM_ST = 0, TM_AB = 128, TM_W = 288, TM_U = 352, TM_O = 416;
constexpr uint32_t WAIT_LIMIT = 1u << 24;

__device__ __forceinline__ void st_bf16x2(unsigned char *base, uint32_t off, float a, float b) {
    *reinterpret_cast<uint32_t *>(base + off) = pack_bf16(a, b);
}

// Tensor maps of the chunk loads: q, k, g as plain [64 tokens][128] boxes,
// v as two 64-wide halves with the 128-byte swizzle (the MN-major operand
// layout of the U~ product, atoms ordered [half][k group]).
struct TcParams {
    ChunkArgs a;
    CUtensorMap tq, tk, tg, tv;
};

__global__ void __launch_bounds__(NT, 1) kda_chunk_tc_kernel(const __grid_constant__ TcParams P) {
    const ChunkArgs &p = P.a;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte aligned base for the swizzled operand tiles; an offset from the
    // __shared__ array (not an integer round trip) keeps accesses in the
    // shared state space
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(sm);
    const uint32_t sb4 = sb >> 4;  // 16-byte units, for matrix descriptors
    float *sBeta = reinterpret_cast<float *>(sm + OFF_BETA);
    float *sPart = reinterpret_cast<float *>(sm + OFF_PART);
    float *sDel = reinterpret_cast<float *>(sm + OFF_DEL);
    float *sGam = reinterpret_cast<float *>(sm + OFF_GAM);
    const uint32_t bar0 = sb + OFF_BAR;
    uint32_t *sTmem = reinterpret_cast<uint32_t *>(sm + OFF_TMEM);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x, h = blockIdx.y, tile = blockIdx.z;
    const int H = p.H, dv = p.dv;

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
    } else {
        n = 0;
        t0 = unit * p.seg_len;
        t1 = min(p.T, t0 + p.seg_len);
        last_seg = t1 == p.T;
    }
    // start of this unit's sequence (checkpoint positions are relative to it)
    const int seq0 = (p.mode == MODE_SEQ) ? t0 : ((p.seg_table && p.cu_seqlens) ? p.cu_seqlens[n] : 0);
    const bool transition = p.mode == MODE_TRANSITION;
    const bool m_part = transition && tile == 0;  // augmented columns [0, dk): M
    const bool has_v = !m_part;
    const bool need_q = !transition;
    const int vcol0 = transition ? 0 : tile * D;

    // ---------------------------------------------------------------- setup
    if (tid == 0) {
        for (int b = 0; b < 6; ++b) umma::mbar_init(bar0 + 8 * b, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == 0) umma::tmem_alloc(sb + OFF_TMEM, 512);
    umma::fence_before();
    __syncthreads();
    umma::fence_after();
    const uint32_t tmem = *sTmem;

    const int qd = warp & 3, cg = warp >> 2;  // TMEM lane quadrant, column group
    const int jrow = 32 * qd + lane;          // S^T row (value column j) owned
    const uint32_t tq = tmem + ((uint32_t)(32 * qd) << 16);

    {
    float Sreg[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) {
        const int i = 32 * cg + c;
        float v0 = 0.f;
        if (transition) {
            v0 = (m_part && i == jrow) ? 1.f : 0.f;
        } else {
            const float *src = (p.mode == MODE_SEQ) ? p.S_init : p.S_in;
            if (src) {
                size_t sidx = (p.mode == MODE_SEQ) ? (size_t)n : (size_t)unit;
                v0 = src[((sidx * H + h) * D + i) * (size_t)dv + vcol0 + jrow];
            }
        }
        Sreg[c] = v0;
    }
    umma::st32(tq + TM_ST + 32 * cg, Sreg);
    }

    const float g_min = p.g_min;

    const uint32_t bar_qkg = bar0 + 32, bar_v = bar0 + 40;
    // one thread issues the bulk copies of a chunk; rows past the end of the
    // tensor are zero-filled by the copy engine, rows past the end of the
    // segment are zeroed after arrival (fix_tail)
    auto issue_qkg = [&](int tc) {
        if (tid == 0) {
            umma::fence_proxy_async();
            umma::mbar_expect_tx(bar_qkg, (need_q ? 16384u : 0u) + 16384u + 32768u);
            if (need_q) umma::tma_load_3d(sb + OFF_Q, &P.tq, 0, h, tc, bar_qkg);
            umma::tma_load_3d(sb + OFF_K, &P.tk, 0, h, tc, bar_qkg);
            umma::tma_load_3d(sb + OFF_G, &P.tg, 0, h, tc, bar_qkg);
        }
    };
    // values: consumed up to the W / U~ products (step 6), so they are
    // prefetched after those, separately from q, k, g (consumed in step 2)
    auto issue_v = [&](int tc) {
        if (tid == 0 && has_v) {
            umma::fence_proxy_async();
            umma::mbar_expect_tx(bar_v, 16384u);
            umma::tma_load_3d(sb + OFF_V, &P.tv, vcol0, h, tc, bar_v);
            umma::tma_load_3d(sb + OFF_V + 8192, &P.tv, vcol0 + 64, h, tc, bar_v);
        }
    };
    auto load_beta = [&](int tc) -> float {
        const int Lc = min(CH, t1 - tc);
        return (tid < Lc) ? p.beta[(size_t)(tc + tid) * H + h] : 0.f;
    };
    if (!has_v) {  // the M part of a transition walks v = 0
        for (int idx = tid; idx < 16384 / 16; idx += NT)
            *reinterpret_cast<uint4 *>(sm + OFF_V + idx * 16) = make_uint4(0u, 0u, 0u, 0u);
        umma::fence_proxy_async();
    }

    bool timed_out = false;
    uint32_t phase = 0;
    float beta_next = 0.f;
    uint32_t pending = 0;  // bulk copies issued for the chunk after the current one
    // waits of the current chunk that gave up: bits 0-3 the product barriers
    // bar0 + 8 i, bit 4 the q/k/g copies, bit 5 the v copies
    uint32_t stuck = 0;
    auto wait_or_mark = [&](uint32_t bar, uint32_t bit) {
        if (!umma::mbar_wait(bar, phase, WAIT_LIMIT)) {
            timed_out = true;
            stuck |= bit;
        }
    };
    if (t0 < t1) {
        issue_qkg(t0);
        issue_v(t0);
        if (tid < CH) beta_next = load_beta(t0);
    }

    for (int tc = t0; tc < t1; tc += CH, phase ^= 1u) {
        const int Lc = min(CH, t1 - tc);
        if (tid < CH) sBeta[tid] = beta_next;
        pending = 0;
        wait_or_mark(bar_qkg, 16u);
        if (has_v) wait_or_mark(bar_v, 32u);
        if (Lc < CH) {  // last chunk of the segment: rows past its end are not ours
            for (int idx = tid; idx < (CH - Lc) * 16; idx += NT) {
                const int r = Lc + (idx >> 4), c = idx & 15;
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4 *>(sm + OFF_Q + r * 256 + c * 16) = z;
                *reinterpret_cast<uint4 *>(sm + OFF_K + r * 256 + c * 16) = z;
                *reinterpret_cast<uint4 *>(sm + OFF_G + r * 512 + c * 16) = z;
                *reinterpret_cast<uint4 *>(sm + OFF_G + r * 512 + 256 + c * 16) = z;
                // V rows (token r) in both 64-wide halves: 8 chunks of 16 bytes each
                *reinterpret_cast<uint4 *>(sm + OFF_V + (c >> 3) * 8192 + umma::mnmaj(8 * (c & 7), r, 1)) = z;
            }
            umma::fence_proxy_async();
        }
        if (__syncthreads_or(timed_out)) break;

        // ------------------------------------------------------------ step 2: decays and operands
        {
            const int c2 = tid & 63, i = (tid >> 6) & 3, hf = tid >> 8;
            const int ch = 2 * c2;
            const int tb = 16 * i + 8 * hf;
            float2 e[8], xl[8], yl[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                float2 gv = *reinterpret_cast<const float2 *>(sm + OFF_G + (tb + r) * 512 + ch * 4);
                e[r].x = __expf(fmaxf(gv.x, g_min));
                e[r].y = __expf(fmaxf(gv.y, g_min));
            }
            float2 pr = make_float2(1.f, 1.f);
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                pr.x *= e[r].x;
                pr.y *= e[r].y;
                xl[r] = pr;
            }
            float2 sf = make_float2(1.f, 1.f);
#pragma unroll
            for (int r = 7; r >= 0; --r) {
                yl[r] = sf;
                sf.x *= e[r].x;
                sf.y *= e[r].y;
            }
            *reinterpret_cast<float2 *>(sPart + (hf * 4 + i) * 128 + ch) = pr;
            __syncthreads();
            const float2 p0 = *reinterpret_cast<const float2 *>(sPart + (0 * 4 + i) * 128 + ch);
            const float2 p1 = *reinterpret_cast<const float2 *>(sPart + (1 * 4 + i) * 128 + ch);
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                if (hf == 0) {
                    yl[r].x *= p1.x;
                    yl[r].y *= p1.y;
                } else {
                    xl[r].x *= p0.x;
                    xl[r].y *= p0.y;
                }
            }
            if (hf == 0) *reinterpret_cast<float2 *>(sDel + i * 128 + ch) = make_float2(p0.x * p1.x, p0.y * p1.y);
            __syncthreads();
            float2 dl[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) dl[m] = *reinterpret_cast<const float2 *>(sDel + m * 128 + ch);
            float2 gb = make_float2(1.f, 1.f), cc = make_float2(1.f, 1.f);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                if (m < i) { gb.x *= dl[m].x; gb.y *= dl[m].y; }
                if (m > i) { cc.x *= dl[m].x; cc.y *= dl[m].y; }
            }
            if (i == 0 && hf == 0) {
                *reinterpret_cast<float2 *>(sGam + ch) = make_float2(
                    ((dl[0].x * dl[1].x) * dl[2].x) * dl[3].x, ((dl[0].y * dl[1].y) * dl[2].y) * dl[3].y);
            }
            // right-operand factors for row blocks i2 >= i: 1/delta_i (i2 == i), c_{i2,i} otherwise
            float2 vf[4];
#pragma unroll
            for (int i2 = 0; i2 < 4; ++i2) {
                float2 f = make_float2(1.f, 1.f);
                if (i2 == i) {
                    f = make_float2(__frcp_rn(dl[i].x), __frcp_rn(dl[i].y));
                } else {
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        if (m > i && m < i2) { f.x *= dl[m].x; f.y *= dl[m].y; }
                }
                vf[i2] = f;
            }
            // Every destination row of this thread's token r has (row & 7) == r,
            // so one swizzled column offset per r serves all operands; row bases
            // are per-thread constants.
            const uint32_t c8 = (uint32_t)(ch & 63) >> 3, lo = (uint32_t)(ch & 7) << 1, kb = (uint32_t)ch >> 6;
            const uint32_t rowL = (uint32_t)(32 * i + 8 * hf) * 128u;  // key rows; query rows +2048
            const uint32_t rowT = (uint32_t)tb * 128u;                 // token rows
            const uint32_t un = sb + OFF_UN;
            const uint32_t aL = un + UN_L + kb * 16384u + rowL;
            const uint32_t aQT = sb + OFF_QT + kb * 8192u + rowT;
            const uint32_t atom = ((uint32_t)(2 * i + hf) * 2u + kb) * 1024u;
            const uint32_t aKG = sb + OFF_KG + atom;
            const uint32_t aKT = sb + OFF_KT + atom;
            const uint32_t aRk = un + UN_R + kb * R_KB + rowT;
            const uint32_t aR0 = aRk + r_row(0) * 128u, aR1 = aRk + r_row(1) * 128u;
            const uint32_t aR2 = aRk + r_row(2) * 128u, aR3 = aRk + r_row(3) * 128u;
            const uint32_t ak = sb + OFF_K + rowT * 2u + (uint32_t)ch * 2u;  // raw rows are 256 B
            const uint32_t aq = sb + OFF_Q + rowT * 2u + (uint32_t)ch * 2u;
            uint32_t kraw[8], qraw[8];  // loads first: the stores below are ordered asm
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                kraw[r] = lds32(ak + r * 256);
                qraw[r] = need_q ? lds32(aq + r * 256) : 0u;
            }
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const uint32_t o = (uint32_t)r * 128u + ((c8 ^ (uint32_t)r) << 4) + lo;
                const float2 kv = unpack_bf16(kraw[r]);
                const float2 x = xl[r], y = yl[r];
                const float2 lk = make_float2(kv.x * x.x, kv.y * x.y);
                const float2 ky = make_float2(kv.x * y.x, kv.y * y.y);
                sts32(aL + o, pack_bf16(lk.x, lk.y));
                if (i <= 0) sts32(aR0 + o, pack_bf16(ky.x * vf[0].x, ky.y * vf[0].y));
                if (i <= 1) sts32(aR1 + o, pack_bf16(ky.x * vf[1].x, ky.y * vf[1].y));
                if (i <= 2) sts32(aR2 + o, pack_bf16(ky.x * vf[2].x, ky.y * vf[2].y));
                sts32(aR3 + o, pack_bf16(ky.x * vf[3].x, ky.y * vf[3].y));
                sts32(aKG + o, pack_bf16(lk.x * gb.x, lk.y * gb.y));
                sts32(aKT + o, pack_bf16(ky.x * cc.x, ky.y * cc.y));
                if (need_q) {
                    const float2 qv = unpack_bf16(qraw[r]);
                    const float2 lq = make_float2(qv.x * x.x, qv.y * x.y);
                    sts32(aL + 2048 + o, pack_bf16(lq.x, lq.y));
                    sts32(aQT + o, pack_bf16(lq.x * gb.x, lq.y * gb.y));
                }
            }
        }
        umma::fence_proxy_async();
        __syncthreads();

        // ------------------------------------------------------------ step 3: A and B tiles
        // D[t'][s'] = L[t'] . R[s'] over all 128 L rows and 160 R rows in one
        // M = 128, N = 160 product: block i reads its 32 L rows (TMEM lane
        // quadrant i) against its R_i columns; the other pairs are not used
        if (tid == 0) {
            umma::fence_after();
            constexpr uint32_t id = umma::idesc_bf16(128, 160, 0, 0, 0);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t kb = ks >> 2, kin = (ks & 3) * 32;
                const uint64_t a = umma::sdesc4(sb4 + ((OFF_UN + UN_L + kb * 16384 + kin) >> 4), 16, 1024);
                const uint64_t b = umma::sdesc4(sb4 + ((OFF_UN + UN_R + kb * R_KB + kin) >> 4), 16, 1024);
                umma::mma(tmem + TM_AB, a, b, id, ks > 0 ? 1u : 0u);
            }
            umma::commit(bar0 + 0);
        }
        if (tc + CH < t1) {  // raw q, k, g consumed: prefetch the next chunk's
            issue_qkg(tc + CH);
            pending |= 1u;
        }
        wait_or_mark(bar0 + 0, 1u);
        umma::fence_after();

        // S^T (rows of this thread's TMEM lane, columns 32 cg ..) as the bf16
        // operand of steps 6 and 8, and the resident state decayed to the chunk
        // end in place, Diag-cols(e^{gamma_63}) S^T, onto which step 10 accumulates
        // U^T K~.  Done in step 4 or step 5 (see early_copy).
        auto copy_decay_state = [&]() {
            float Sreg[32];
            umma::ld32(tq + TM_ST + 32 * cg, Sreg);
#pragma unroll
            for (int c = 0; c < 32; c += 8) {
                uint4 pk;
                pk.x = pack_bf16(Sreg[c + 0], Sreg[c + 1]);
                pk.y = pack_bf16(Sreg[c + 2], Sreg[c + 3]);
                pk.z = pack_bf16(Sreg[c + 4], Sreg[c + 5]);
                pk.w = pack_bf16(Sreg[c + 6], Sreg[c + 7]);
                *reinterpret_cast<uint4 *>(sm + OFF_UN + UN_ST + umma::kmaj(jrow, 32 * cg + c, 128)) = pk;
            }
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
                const float4 gm = *reinterpret_cast<const float4 *>(sGam + 32 * cg + c);
                Sreg[c + 0] *= gm.x;
                Sreg[c + 1] *= gm.y;
                Sreg[c + 2] *= gm.z;
                Sreg[c + 3] *= gm.w;
            }
            umma::st32(tq + TM_ST + 32 * cg, Sreg);
            umma::fence_before();
        };

        // half of the warps copy the state in step 4: those without A/B columns
        // there (cg > lane quadrant) and warps 2, 3 (busy in step 5)
        const bool early_copy = cg > qd || warp == 2 || warp == 3;

        // ------------------------------------------------------------ step 4: A (fp32, scaled by b_t) and B (bf16)
        // Lane quadrant i holds block i: lanes 0-15 the key rows t = 16 i + l (A),
        // 16-31 the query rows (B); warp (i, cg) takes key columns s = 16 cg ..
        // 16 cg + 15 of R_i when cg <= i, else those entries are zero.
        {
            float *sAf = reinterpret_cast<float *>(sm + OFF_UN + UN_AF);
            const int i = qd, t = 16 * i + (lane & 15), s0 = 16 * cg;
            const bool is_q = lane >= 16;
            float v[16];
            if (cg <= i) umma::ld16(tq + TM_AB + r_row(i) + 16 * cg, v);
            else {
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = 0.f;
            }
            if (!is_q) {
                if (cg <= i) {
                    const float bt = sBeta[t];
#pragma unroll
                    for (int j = 0; j < 16; j += 4)
                        *reinterpret_cast<float4 *>(sAf + t * LDF + s0 + j) =
                            make_float4((s0 + j < t) ? bt * v[j] : 0.f, (s0 + j + 1 < t) ? bt * v[j + 1] : 0.f,
                                        (s0 + j + 2 < t) ? bt * v[j + 2] : 0.f, (s0 + j + 3 < t) ? bt * v[j + 3] : 0.f);
                }
            } else {
                uint32_t bp[8];
#pragma unroll
                for (int j = 0; j < 16; j += 2)
                    bp[j >> 1] = pack_bf16((s0 + j <= t) ? v[j] : 0.f, (s0 + j + 1 <= t) ? v[j + 1] : 0.f);
                // B as a K-major operand: row t, k = s
                const uint32_t row = (uint32_t)t * 128u, sw = (uint32_t)(t & 7);
                *reinterpret_cast<uint4 *>(sm + OFF_BM + row + (((2u * cg) ^ sw) << 4)) =
                    make_uint4(bp[0], bp[1], bp[2], bp[3]);
                *reinterpret_cast<uint4 *>(sm + OFF_BM + row + (((2u * cg + 1u) ^ sw) << 4)) =
                    make_uint4(bp[4], bp[5], bp[6], bp[7]);
            }
            if (early_copy) copy_decay_state();
        }
        if (__syncthreads_or(timed_out)) break;

        // ------------------------------------------------------------ step 5: T = (I + A)^{-1}, fp32
        {
            const float *sAf = reinterpret_cast<const float *>(sm + OFF_UN + UN_AF);
            float *sTf = reinterpret_cast<float *>(sm + OFF_UN + UN_TF);
            // diagonal 16 x 16 blocks, right-looking substitution with one column
            // per lane in registers: lanes 0-15 of warp 2 + w -> block 2w, 16-31 -> 2w+1
            if (!early_copy) copy_decay_state();
            if (warp == 2 || warp == 3) {
                const int i = 2 * (warp - 2) + (lane >> 4), c = lane & 15;
                const float *Ab = sAf + (16 * i) * LDF + 16 * i;
                float acc[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) acc[r] = (r == c) ? 1.f : 0.f;
#pragma unroll
                for (int m = 0; m < 15; ++m) {
                    const float cm = acc[m];
#pragma unroll
                    for (int r = m + 1; r < 16; ++r) acc[r] = fmaf(-Ab[r * LDF + m], cm, acc[r]);
                }
                float *Tb = sTf + (16 * i) * LDF + 16 * i;
#pragma unroll
                for (int r = 0; r < 16; ++r) Tb[r * LDF + c] = acc[r];
            }
            __syncthreads();
            // 32 x 32 diagonal halves: T_10 = -T_11 A_10 T_00, T_32 = -T_33 A_32 T_22.
            // X = A_10 T_00 goes to the (unused) upper block (0,1) of the A scratch.
            {
                const int hb = tid >> 8, e = tid & 255, r = e >> 4, c = e & 15;
                const int i = 2 * hb + 1, j = 2 * hb;
                const float *Ar = sAf + (16 * i + r) * LDF + 16 * j;
                const float *Tc = sTf + (16 * j) * LDF + 16 * j + c;
                float x0 = 0.f, x1 = 0.f;
#pragma unroll
                for (int m = 0; m < 16; m += 2) {
                    x0 = fmaf(Ar[m], Tc[m * LDF], x0);
                    x1 = fmaf(Ar[m + 1], Tc[(m + 1) * LDF], x1);
                }
                float *Xs = const_cast<float *>(sAf) + (16 * j) * LDF + 16 * i;  // X[r][c] at row r
                Xs[r * LDF + c] = x0 + x1;
                // the upper blocks (0,1) and (2,3) of T are zero (read as parts of the
                // lower-triangular 32 x 32 halves below)
                sTf[(16 * j + r) * LDF + 16 * i + c] = 0.f;
                __syncthreads();
                const float *Ti = sTf + (16 * i + r) * LDF + 16 * i;
                float y0 = 0.f, y1 = 0.f;
#pragma unroll
                for (int m = 0; m < 16; m += 2) {
                    y0 = fmaf(Ti[m], Xs[m * LDF + c], y0);
                    y1 = fmaf(Ti[m + 1], Xs[(m + 1) * LDF + c], y1);
                }
                sTf[(16 * i + r) * LDF + 16 * j + c] = -(y0 + y1);
                __syncthreads();
            }
            // Warps 0-7: lower-left 32 x 32, T_21 = -T_22 (A_21 T_11), two 32x32x32
            // fp32 products as tf32 tensor products with hi/lo splits (3 MMAs per
            // step); warp w owns the 16 x 8 tile (rows 16(w>>2), cols 8(w&3)); the
            // intermediate X goes to the unused upper-right 32 x 32 of the A scratch
            // and the result straight into T diag(b) as bf16.
            // Warps 8-15 meanwhile: T diag(b) for the rest (rows 0-31 and the
            // lower-right 32 x 32), zero above the diagonal.
            if (warp < 8) {
                const int gq = lane >> 2, q4 = lane & 3;
                const int mt = (warp >> 2) & 1, nt = warp & 3;
                auto product = [&](const float *Am, const float *Bm, float (&acc)[4]) {
                    acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        uint32_t ah[4], al[4], bh0, bl0, bh1, bl1;
                        split_tf32(Am[(16 * mt + gq) * LDF + 8 * kk + q4], ah[0], al[0]);
                        split_tf32(Am[(16 * mt + gq + 8) * LDF + 8 * kk + q4], ah[1], al[1]);
                        split_tf32(Am[(16 * mt + gq) * LDF + 8 * kk + q4 + 4], ah[2], al[2]);
                        split_tf32(Am[(16 * mt + gq + 8) * LDF + 8 * kk + q4 + 4], ah[3], al[3]);
                        split_tf32(Bm[(8 * kk + q4) * LDF + 8 * nt + gq], bh0, bl0);
                        split_tf32(Bm[(8 * kk + q4 + 4) * LDF + 8 * nt + gq], bh1, bl1);
                        mma_tf32(acc, al, bh0, bh1);
                        mma_tf32(acc, ah, bl0, bl1);
                        mma_tf32(acc, ah, bh0, bh1);
                    }
                };
                float acc[4];
                float *X64 = const_cast<float *>(sAf) + 32;  // rows 0-31, columns 32-63
                product(sAf + 32 * LDF, sTf, acc);           // X = A_21 T_11
                float *Xt = X64 + (16 * mt + gq) * LDF + 8 * nt + 2 * q4;
                *reinterpret_cast<float2 *>(Xt) = make_float2(acc[0], acc[1]);
                *reinterpret_cast<float2 *>(Xt + 8 * LDF) = make_float2(acc[2], acc[3]);
                asm volatile("bar.sync 1, 256;\n" ::: "memory");  // warps 0-7 only
                product(sTf + 32 * LDF + 32, X64, acc);      // T_22 X
                const int t = 32 + 16 * mt + gq, s0 = 8 * nt + 2 * q4;
                const float b0 = sBeta[s0], b1 = sBeta[s0 + 1];
                st_bf16x2(sm, OFF_TB + umma::kmaj(t, s0, 64), -acc[0] * b0, -acc[1] * b1);
                st_bf16x2(sm, OFF_TB + umma::kmaj(t + 8, s0, 64), -acc[2] * b0, -acc[3] * b1);
            } else {
                // 1536 pairs: rows 0-31 x 32 pairs, then rows 32-63 x pairs 16-31
                for (int e2 = tid - 256; e2 < 1536; e2 += 256) {
                    int t, s;
                    if (e2 < 1024) {
                        t = e2 >> 5;
                        s = 2 * (e2 & 31);
                    } else {
                        t = 32 + ((e2 - 1024) >> 4);
                        s = 32 + 2 * ((e2 - 1024) & 15);
                    }
                    const float a0 = (s <= t) ? sTf[t * LDF + s] * sBeta[s] : 0.f;
                    const float a1 = (s + 1 <= t) ? sTf[t * LDF + s + 1] * sBeta[s + 1] : 0.f;
                    st_bf16x2(sm, OFF_TB + umma::kmaj(t, s, 64), a0, a1);
                }
            }
        }
        umma::fence_proxy_async();
        __syncthreads();

        // ------------------------------------------------------------ step 6: W^T and U~^T
        if (tid == 0) {
            umma::fence_after();
            constexpr uint32_t id = umma::idesc_bf16(128, 64, 1, 0, 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint64_t b = umma::sdesc4(sb4 + ((OFF_TB + ks * 32) >> 4), 16, 1024);
                umma::mma(tmem + TM_W, umma::sdesc4(sb4 + ((OFF_KG + ks * 4096) >> 4), 1024, 2048), b, id, ks > 0 ? 1u : 0u);
                if (has_v)  // V halves are 8 KB apart (LBO), k groups 1 KB apart (SBO)
                    umma::mma(tmem + TM_U, umma::sdesc4(sb4 + ((OFF_V + ks * 2048) >> 4), 8192, 1024), b, id, ks > 0 ? 1u : 0u);
            }
            umma::commit(bar0 + 8);
            // S^T Q~^T needs only the state copy and Q~: it runs behind W / U~ and
            // completes under step 8's commit
            if (need_q) {
                constexpr uint32_t idq = umma::idesc_bf16(128, 64, 0, 0, 0);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t kb = ks >> 2, kin = (ks & 3) * 32;
                    umma::mma(tmem + TM_O, umma::sdesc4(sb4 + ((OFF_UN + UN_ST + kb * 16384 + kin) >> 4), 16, 1024),
                              umma::sdesc4(sb4 + ((OFF_QT + kb * 8192 + kin) >> 4), 16, 1024), idq, ks > 0 ? 1u : 0u);
                }
            }
        }
        wait_or_mark(bar0 + 8, 2u);
        umma::fence_after();
        if (tc + CH < t1) {  // V and b consumed: prefetch the next chunk's
            issue_v(tc + CH);
            pending |= 2u;
            if (tid < CH) beta_next = load_beta(tc + CH);
        }

        // ------------------------------------------------------------ step 7: W (bf16) operand
        {
            float v[16];
            umma::ld16(tq + TM_W + 16 * cg, v);
            const int i = jrow;  // key channel
            // W as an MN-major operand: element (n = t, k = i), t contiguous
            *reinterpret_cast<uint4 *>(sm + OFF_UN + UN_W + umma::mnmaj(16 * cg, i, 1)) =
                make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
            *reinterpret_cast<uint4 *>(sm + OFF_UN + UN_W + umma::mnmaj(16 * cg + 8, i, 1)) =
                make_uint4(pack_bf16(v[8], v[9]), pack_bf16(v[10], v[11]), pack_bf16(v[12], v[13]),
                           pack_bf16(v[14], v[15]));
        }
        umma::fence_proxy_async();
        umma::fence_before();
        if (__syncthreads_or(timed_out)) break;

        // ------------------------------------------------------------ step 8: U~^T - S^T W^T
        if (tid == 0) {
            umma::fence_after();
            constexpr uint32_t idw = umma::idesc_bf16(128, 64, 0, 1, 1);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t kb = ks >> 2, kin = (ks & 3) * 32;
                const uint64_t a = umma::sdesc4(sb4 + ((OFF_UN + UN_ST + kb * 16384 + kin) >> 4), 16, 1024);
                umma::mma(tmem + TM_U, a, umma::sdesc4(sb4 + ((OFF_UN + UN_W + ks * 2048) >> 4), 1024, 1024), idw,
                          (has_v || ks > 0) ? 1u : 0u);
            }
            umma::commit(bar0 + 16);
        }
        wait_or_mark(bar0 + 16, 4u);
        umma::fence_after();

        // ------------------------------------------------------------ step 9: U^T (bf16) operand
        {
            float v[16];
            umma::ld16(tq + TM_U + 16 * cg, v);
#pragma unroll
            for (int c = 0; c < 16; c += 8) {
                uint4 pk;
                pk.x = pack_bf16(v[c + 0], v[c + 1]);
                pk.y = pack_bf16(v[c + 2], v[c + 3]);
                pk.z = pack_bf16(v[c + 4], v[c + 5]);
                pk.w = pack_bf16(v[c + 6], v[c + 7]);
                *reinterpret_cast<uint4 *>(sm + OFF_UN + UN_UT + umma::kmaj(jrow, 16 * cg + c, 128)) = pk;
            }
        }
        umma::fence_proxy_async();
        umma::fence_before();
        if (__syncthreads_or(timed_out)) break;

        // ------------------------------------------------------------ step 10: + U^T B^T, U^T K~
        if (tid == 0) {
            umma::fence_after();
            constexpr uint32_t ido = umma::idesc_bf16(128, 64, 0, 0, 0);
            constexpr uint32_t ids = umma::idesc_bf16(128, 128, 0, 1, 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint64_t a = umma::sdesc4(sb4 + ((OFF_UN + UN_UT + ks * 32) >> 4), 16, 1024);
                if (need_q) umma::mma(tmem + TM_O, a, umma::sdesc4(sb4 + ((OFF_BM + ks * 32) >> 4), 16, 1024), ido, 1u);
                umma::mma(tmem + TM_ST, a, umma::sdesc4(sb4 + ((OFF_KT + ks * 4096) >> 4), 1024, 2048), ids, 1u);
            }
            umma::commit(bar0 + 24);
        }
        wait_or_mark(bar0 + 24, 8u);
        umma::fence_after();
        // checkpoint: the state after token (tc + Lc) when that position of the
        // sequence is a multiple of ckpt_every (S^T lane = value column)
        if (p.ckpt && !transition) {
            const int rel = tc + Lc - seq0;
            const int kq = rel / p.ckpt_every - 1;
            if (rel % p.ckpt_every == 0 && kq < p.ckpt_count) {
                float *dst = p.ckpt + (((size_t)n * p.ckpt_count + kq) * H + h) * D * (size_t)dv;
                float Sreg[32];
                umma::ld32(tq + TM_ST + 32 * cg, Sreg);
#pragma unroll
                for (int c = 0; c < 32; ++c) dst[(size_t)(32 * cg + c) * dv + vcol0 + jrow] = Sreg[c];
            }
        }

        // ------------------------------------------------------------ step 11: outputs and state
        // outputs are staged as a row-major [64][128] bf16 tile in the (now free)
        // union region, then written with 16-byte stores
        unsigned char *ostage = sm + OFF_UN;
        if (need_q) {
            float v[16];
            umma::ld16(tq + TM_O + 16 * cg, v);
#pragma unroll
            for (int tt = 0; tt < 16; ++tt)
                *reinterpret_cast<__nv_bfloat16 *>(ostage + (16 * cg + tt) * 256 + jrow * 2) =
                    __float2bfloat16_rn(p.scale * v[tt]);
        }
        umma::fence_before();
        if (__syncthreads_or(timed_out)) break;
        if (need_q) {
            __nv_bfloat16 *og = reinterpret_cast<__nv_bfloat16 *>(p.o);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int idx = tid + u * NT, t = idx >> 4, c = idx & 15;
                if (t < Lc)
                    *reinterpret_cast<uint4 *>(og + ((size_t)(tc + t) * H + h) * dv + vcol0 + c * 8) =
                        *reinterpret_cast<const uint4 *>(ostage + t * 256 + c * 16);
            }
        }
    }

    if (timed_out) {
        if (tid == 0) report_status(p.status, KDA_STATUS_TIMEOUT);
        // let copies still in flight land and products still running finish
        // before the shared and tensor memory are released
        for (int i = 0; i < 4; ++i)
            if (stuck & (1u << i)) umma::mbar_wait(bar0 + 8 * i, phase, WAIT_LIMIT);
        if (stuck & 16u) umma::mbar_wait(bar_qkg, phase, WAIT_LIMIT);
        if (stuck & 32u) umma::mbar_wait(bar_v, phase, WAIT_LIMIT);
        if (pending & 1u) umma::mbar_wait(bar_qkg, phase ^ 1u, WAIT_LIMIT);
        if ((pending & 2u) && has_v) umma::mbar_wait(bar_v, phase ^ 1u, WAIT_LIMIT);
    } else {
        // ------------------------------------------------------------ state out
        float *dst = nullptr;
        size_t ld_dst = (size_t)dv, col0 = (size_t)vcol0;
        if (p.mode == MODE_SEQ) {
            if (p.S_final) dst = p.S_final + ((size_t)n * H + h) * D * (size_t)dv;
        } else if (p.mode == MODE_REPLAY) {
            if (p.S_final && last_seg) dst = p.S_final + ((size_t)n * H + h) * D * (size_t)dv;
        } else if (m_part) {
            dst = p.M_out + ((size_t)unit * H + h) * D * (size_t)D;
            ld_dst = D;
            col0 = 0;
        } else {
            dst = p.N_out + ((size_t)unit * H + h) * D * (size_t)dv;
            col0 = 0;
        }
        if (dst) {
            float Sreg[32];
            umma::ld32(tq + TM_ST + 32 * cg, Sreg);
#pragma unroll
            for (int c = 0; c < 32; ++c) dst[(size_t)(32 * cg + c) * ld_dst + col0 + jrow] = Sreg[c];
        }
    }
    umma::fence_before();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(tmem, 512);
}

}  // namespace tc

void *tensor_map_encoder() {
    static void *fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = ptr;
    }
    return fn;
}

bool chunk_tc_supported(const ChunkArgs &a, bool in_bf16) {
    return in_bf16 && a.dk == 128 && a.dv == 128;
}

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() { return reinterpret_cast<EncodeTiledFn>(tensor_map_encoder()); }

// [T][H][inner] tensor, box of `box_inner` x 1 head x 64 tokens
bool make_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize, int inner, int H, int T,
              int box_inner, CUtensorMapSwizzle swz) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)H, (cuuint64_t)(T > 0 ? T : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)inner * esize, (cuuint64_t)inner * esize * H};
    cuuint32_t box[3] = {(cuuint32_t)box_inner, 1u, 64u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    return fn(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

cudaError_t launch_chunk_tc(const ChunkArgs &a, int units, cudaStream_t st) {
    const int ntiles = (a.mode == MODE_TRANSITION) ? 2 : 1;
    if (units <= 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(tc::kda_chunk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         tc::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    tc::TcParams P;
    memset(&P, 0, sizeof(P));
    P.a = a;
    const int T = a.T;
    bool ok = make_map(&P.tk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 128, a.H, T, 128, CU_TENSOR_MAP_SWIZZLE_NONE) &&
              make_map(&P.tg, a.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 128, a.H, T, 128, CU_TENSOR_MAP_SWIZZLE_NONE) &&
              make_map(&P.tv, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.dv, a.H, T, 64, CU_TENSOR_MAP_SWIZZLE_128B);
    if (ok && a.q) ok = make_map(&P.tq, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 128, a.H, T, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!ok) return cudaErrorInvalidValue;
    dim3 grid(units, a.H, ntiles);
    tc::kda_chunk_tc_kernel<<<grid, tc::NT, tc::SMEM_BYTES, st>>>(P);
    return cudaGetLastError();
}

}  // namespace kda
