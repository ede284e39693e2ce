// chunk_bwd_tc.cu -- backward of the tensor-core prefill (dk = dv = 128, bf16
// inputs) in the chunk (WY) form: the chunk kernel's training use ("Noyaux KDA
// et FlashKDA", section "FlashKDA : le noyau par blocs").
//
// For a 64-token chunk entered with state S (gamma the running sum of the
// floored log-decays per key channel, Gam = e^gamma, Gam_C its last value,
// K~ = K Gam, Q~ = Q Gam, K^ = K Gam_C / Gam, M = strict_lower(K~ (K / Gam)^T),
// A = diag(b) M, T = (I + A)^{-1}, TB = T diag(b), W = TB K~):
//     Vres = V - K~ S,  U = TB Vres,  O = scale (Q~ S + B U),
//     S_C = diag(Gam_C) S + K^^T U.
// Only the state gradient dS_C (arriving at the chunk end) is serial; it is
// the adjoint of the forward walk on the same operand blobs:
//     dU = scale B^T dO + K^ dS_C,  dS = scale Q~^T dO + diag(Gam_C) dS_C - W^T dU.
// Given the chunk-start state S and dS_C, every chunk's token gradients are
// local (the reverse of each forward step):
//     dVres = TB^T dU (= dv),  dTB = dU Vres^T,  dT = dTB diag(b),
//     dbeta_s = sum_t dTB[t][s] T[t][s] + sum_s' dA[s][s'] M[s][s'],
//     dA = strict_lower(-T^T dT T^T) = strict_lower(-(T^T dU) U^T)  (U = T diag(b) Vres),
//     dM = diag(b) dA,  dB = scale lower(dO U^T),
//     dQ~ = scale dO S^T + (dB through the causal tiles),
//     dK~ = -dVres S^T + (dM through the causal tiles),  dK^ = U dS_C^T,
//     dgamma_C += Gam_C . rowsum(dS_C . S)
// and the log-decay gradient is the reverse cumulative sum of the gradient of
// gamma.  The causal tiles M and B carry the forward's 16-token block
// anchoring: row t (block i) is L_t = k_t x_t (x_t = e^{gamma_t - gamma_a},
// a = the token before block i), column s of row block i is
// R_i[s] = k_s e^{gamma_a - gamma_s}; so with A' holding dM and dB in the
// segment columns of each row's block, dL = A' R_seg (rows) and
// dR_seg = A'^T L (columns), both single tensor-core products, and
// dk_t += x_t dL_t, dk_s += sum_i f_i(s) dR_i[s] (f_i(s) = e^{gamma_a_i - gamma_s}),
// dgamma = k . dk-terms with the signs of their exponents.
//
// Three launches after the forward pass (which keeps every blob, the fp32 T
// and M of every chunk, and the walk's bf16 operand tiles S^T and U^T):
//   kda_bwd_walk_kernel   one CTA per (sequence, head), chunks in reverse: dS'
//                         = dS / scale resident in tensor memory, the four
//                         products of a chunk on the tensor cores; keeps the
//                         bf16 tiles dS'^T and dU'^T of every chunk;
//   kda_bwd_chunk_kernel  persistent over (chunk, head) items: three batches
//                         of products per item on the tensor cores (operands in
//                         shared memory, accumulators in tensor memory), the
//                         rest on the CUDA cores in fp32.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_umma.cuh"

namespace kda {
namespace bt {

constexpr int D = 128;
constexpr int CH = 64;
constexpr uint32_t WAIT_LIMIT = 1u << 24;
// The bound of the first wait of each kernel (the reverse walk's on its first
// chunk's copies, the chunk kernel's on its first item's copies).  A test
// build (KDA_TEST_SHORT_FIRST_WAIT) gives up on it at once, to exercise the
// timeout path: status reported, the copies still in flight drained (full
// bound), memory released.  The library itself uses the full bound.
#ifdef KDA_TEST_SHORT_FIRST_WAIT
constexpr uint32_t FIRST_WAIT_LIMIT = 0;
#else
constexpr uint32_t FIRST_WAIT_LIMIT = WAIT_LIMIT;
#endif
constexpr uint32_t TILE_S = 32768;  // bf16 S^T / dS'^T tile (K-major 128 x 128)
constexpr uint32_t TILE_U = 16384;  // bf16 U^T / dU'^T tile (K-major 128 x 64)
constexpr uint32_t AUX_FLOATS = 8192;

// first row of segment i of the anchored column operand: 8 i (i + 1)
__host__ __device__ constexpr int segoff(int i) { return 8 * i * (i + 1); }

__device__ __forceinline__ float bf16_at(const void *base, size_t idx) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(base)[idx]);
}
__device__ __forceinline__ uint16_t bf16_bits(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}
__device__ __forceinline__ float bf16_round(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// ============================================================================ reverse walk
constexpr int NR = 512;
constexpr uint32_t R_BUF = 0;          // two operand blobs (double buffer)
constexpr uint32_t R_BUFSTRIDE = 66560;
constexpr uint32_t R_DO = 133120;      // two dO tiles (value halves of [64 t][128 B], 8 KB apart)
constexpr uint32_t R_ST = 165888;      // dS'^T bf16, K-major 128 x 128
constexpr uint32_t R_UT = 198656;      // dU'^T bf16, K-major 128 x 64
constexpr uint32_t R_BAR = 215040;     // 4 mbarriers: buffer 0, buffer 1, dU product, dS products
constexpr uint32_t R_TMEM = 215072;
constexpr uint32_t R_SMEM = 215088 + 1024;
constexpr uint32_t TM_S = 0, TM_U = 128;  // 256 columns

struct RwalkParams {
    const int32_t *cu;             // [N + 1]
    int N, T, H;
    CUtensorMap tdo;               // dout [T][H][128] bf16, box 64 x 1 x 64, 128-byte swizzle
    const unsigned char *blob;     // [slot][H][kChunkBlobBytes]
    const float *dS_final;         // [N][H][128][128] or null (zero)
    float *dS0;                    // [N][H][128][128] or null
    float wscale;                  // the state gradient walks as dS / wscale
    int zero_do;                   // scale == 0: dO enters no product
    unsigned char *save_ds, *save_du;  // [slot][H] tiles dS'^T (32 KB), dU'^T (16 KB)
    // this launch walks the chunks in slots [slot0, slot1) (a piece); a
    // sequence that continues in later slots starts from carry_in, one that
    // continues in earlier slots leaves its dS' in carry_out ([H][128][128]
    // f32 each, lane-major as the tensor memory holds it)
    int slot0, slot1;
    const float *carry_in;
    float *carry_out;
    // context-parallel segments (seg_table non-null): unit = segment, its
    // token range from the table ({sequence, t0, t1, last} per segment);
    // the walk starts from dS_in[unit][h] (raw dS', [dk][dv]) or from zero
    // when dS_in is null, and leaves the raw dS' at the segment start in
    // r_out[unit][h] when r_out is non-null
    const int32_t *seg_table, *seg_count;
    const float *dS_in;
    float *r_out;
    uint32_t *status;
};

__global__ void __launch_bounds__(NR, 1) kda_bwd_walk_kernel(const __grid_constant__ RwalkParams P) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(sm);
    const uint32_t sb4 = sb >> 4;
    const uint32_t bar0 = sb + R_BAR, bar_u = bar0 + 16, bar_o = bar0 + 24;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = blockIdx.x, h = blockIdx.y, H = P.H;
    // a chunk-gradient launch that follows on the stream as a programmatic
    // dependent may start once every CTA of this walk is resident: it reads
    // only what earlier launches wrote
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const bool segs = P.seg_table != nullptr;
    int t0, t1;
    if (segs) {
        if (n >= *P.seg_count) return;
        const int4 se = reinterpret_cast<const int4 *>(P.seg_table)[n];
        t0 = se.y;
        t1 = se.z;
    } else {
        t0 = P.cu[n];
        t1 = P.cu[n + 1];
    }
    const size_t uoff = ((size_t)n * H + h) * D * D;  // [unit][h] (sequence or segment)
    if (t0 < 0 || t1 < t0 || t1 > P.T) {
        if (tid == 0 && h == 0 && P.slot1 == P.N + P.T / CH) report_status(P.status, KDA_STATUS_BAD_SEQLENS);
        return;
    }
    const int nch = (t1 - t0 + CH - 1) / CH, sbase = t0 / CH + n;
    if (nch == 0) {  // an empty unit passes its gradient through (in the piece of its slot)
        if (sbase >= P.slot0 && sbase < P.slot1) {
            if (segs) {
                if (P.r_out)
                    for (int e = tid; e < D * D; e += NR) P.r_out[uoff + e] = P.dS_in ? P.dS_in[uoff + e] : 0.f;
            } else if (P.dS0) {
                for (int e = tid; e < D * D; e += NR) P.dS0[uoff + e] = P.dS_final ? P.dS_final[uoff + e] : 0.f;
            }
        }
        return;
    }
    const int jb = max(0, P.slot0 - sbase), je = min(nch, P.slot1 - sbase);
    if (jb >= je) return;
    const bool cut_in = je < nch, cut_out = jb > 0;  // continues in later / earlier slots
    const float wscale = P.wscale, inv = 1.0f / wscale;

    if (tid == 0) {
        for (int b = 0; b < 4; ++b) umma::mbar_init(bar0 + 8 * b, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == 0) umma::tmem_alloc(sb + R_TMEM, 256);
    umma::fence_before();
    __syncthreads();
    umma::fence_after();
    const uint32_t tmem = *reinterpret_cast<const uint32_t *>(sm + R_TMEM);
    const int qd = warp & 3, cg = warp >> 2;  // TMEM lane quadrant, column group
    const int jrow = 32 * qd + lane;          // dS'^T row (value column j) owned
    const uint32_t tq = tmem + ((uint32_t)(32 * qd) << 16);

    {  // dS'^T = dS_final^T / wscale (lane j, columns = key channel i), or the carried dS'^T
        float r[32];
        if (cut_in || segs) {  // raw dS' carried from a later piece, given for a segment, or zero
            const float *src = cut_in ? P.carry_in + (size_t)h * D * D : (P.dS_in ? P.dS_in + uoff : nullptr);
#pragma unroll
            for (int c = 0; c < 32; ++c) r[c] = src ? src[(size_t)(32 * cg + c) * D + jrow] : 0.f;
        } else {
            const float *src = P.dS_final ? P.dS_final + uoff : nullptr;
#pragma unroll
            for (int c = 0; c < 32; ++c) r[c] = src ? src[(size_t)(32 * cg + c) * D + jrow] * inv : 0.f;
        }
        umma::st32(tq + TM_S + 32 * cg, r);
    }

    // one thread issues the copies of a chunk: the blob (one bulk copy) and dO
    // (two swizzled value halves; rows past the tensor end are zero-filled,
    // rows past the sequence end are zeroed after arrival)
    auto issue = [&](int j, int b) {
        if (tid == 0) {
            umma::fence_proxy_async();
            const uint32_t bar = bar0 + 8 * b;
            umma::mbar_expect_tx(bar, kChunkBlobBytes + 16384u);
            umma::bulk_load(sb + R_BUF + b * R_BUFSTRIDE, P.blob + ((size_t)(sbase + j) * H + h) * kChunkBlobBytes,
                            kChunkBlobBytes, bar);
            umma::tma_load_3d(sb + R_DO + b * 16384, &P.tdo, 0, h, t0 + CH * j, bar);
            umma::tma_load_3d(sb + R_DO + b * 16384 + 8192, &P.tdo, 64, h, t0 + CH * j, bar);
        }
    };

    bool timed_out = false;
    int pend_b = 0;  // buffer with a copy in flight (the next chunk's, or one whose wait gave up)
    uint32_t pend_ph = 0;
    int pend_m = -1;  // products whose completion wait gave up (0: dU, 1: dS)
    uint32_t pend_mph = 0;
    const bool save = P.save_ds != nullptr;
    issue(je - 1, 0);

    for (int j = je - 1; j >= jb; --j) {
        const int it = je - 1 - j, b = it & 1;
        const uint32_t ph = (uint32_t)(it >> 1) & 1u, pm = (uint32_t)it & 1u;
        const int tc = t0 + CH * j, Lc = min(CH, t1 - tc);
        const uint32_t bb = R_BUF + (uint32_t)b * R_BUFSTRIDE;
        const bool landed = umma::mbar_wait(bar0 + 8 * b, ph, j == je - 1 ? FIRST_WAIT_LIMIT : WAIT_LIMIT);
        timed_out |= !landed;
        pend_b = landed ? -1 : b;
        pend_ph = ph;
        if (j > jb && !timed_out) {
            issue(j - 1, b ^ 1);
            pend_b = b ^ 1;
            pend_ph = (uint32_t)((it + 1) >> 1) & 1u;
        }
        const int z0 = P.zero_do ? 0 : Lc;  // dO rows (tokens) past the sequence end are not ours
        for (int idx = tid; idx < (CH - z0) * 16; idx += NR) {
            const int r = z0 + (idx >> 4), c = idx & 15;
            *reinterpret_cast<uint4 *>(sm + R_DO + b * 16384 + (c >> 3) * 8192 + umma::mnmaj(8 * (c & 7), r, 1)) =
                make_uint4(0u, 0u, 0u, 0u);
        }
        // dS'^T (this thread's lane, columns 32 cg ..) as the bf16 operand, and
        // the resident gradient decayed in place, dS'^T diag(Gam_C), onto
        // which the dO^T Q~ and -dU'^T W products accumulate
        {
            const float *gam = reinterpret_cast<const float *>(sm + bb + kBlobGam);
            float r[32];
            umma::ld32(tq + TM_S + 32 * cg, r);
#pragma unroll
            for (int c = 0; c < 32; c += 8) {
                uint4 pk;
                pk.x = pack_bf16(r[c + 0], r[c + 1]);
                pk.y = pack_bf16(r[c + 2], r[c + 3]);
                pk.z = pack_bf16(r[c + 4], r[c + 5]);
                pk.w = pack_bf16(r[c + 6], r[c + 7]);
                *reinterpret_cast<uint4 *>(sm + R_ST + umma::kmaj(jrow, 32 * cg + c, 128)) = pk;
            }
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
                const float4 gm = *reinterpret_cast<const float4 *>(gam + 32 * cg + c);
                const float2 lo = __fmul2_rn(make_float2(r[c], r[c + 1]), make_float2(gm.x, gm.y));
                const float2 hi = __fmul2_rn(make_float2(r[c + 2], r[c + 3]), make_float2(gm.z, gm.w));
                r[c + 0] = lo.x;
                r[c + 1] = lo.y;
                r[c + 2] = hi.x;
                r[c + 3] = hi.y;
            }
            umma::st32(tq + TM_S + 32 * cg, r);
        }
        umma::fence_proxy_async();
        umma::fence_before();
        if (__syncthreads_or(timed_out)) {
            timed_out = true;
            break;
        }

        // ------------------------------------------------------------ dU'^T = dO^T B + dS'^T K^^T; dS'^T += dO^T Q~
        if (tid == 0) {
            umma::fence_after();
            // A = dO^T (MN-major: value halves 8 KB apart, 8-token groups 1 KB);
            // B = the blob's B read as MN-major (n = key token s, k = query token t)
            constexpr uint32_t id_a = umma::idesc_bf16(128, 64, 1, 1, 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma::mma(tmem + TM_U, umma::sdesc4(sb4 + ((R_DO + b * 16384 + ks * 2048) >> 4), 8192, 1024),
                          umma::sdesc4(sb4 + ((bb + kBlobBM + ks * 2048) >> 4), 1024, 1024), id_a, ks > 0 ? 1u : 0u);
            // A = dS'^T (K-major); B = K^ read as K-major (n = t, k = i: 8-token groups 2 KB apart)
            constexpr uint32_t id_b = umma::idesc_bf16(128, 64, 0, 0, 0);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t kb = ks >> 2, kin = (ks & 3) * 32;
                umma::mma(tmem + TM_U, umma::sdesc4(sb4 + ((R_ST + kb * 16384 + kin) >> 4), 16, 1024),
                          umma::sdesc4(sb4 + ((bb + kBlobKT + kb * 1024 + kin) >> 4), 16, 2048), id_b, 1u);
            }
            umma::commit(bar_u);
            // B = Q~ read as MN-major (n = i: 64-channel blocks 8 KB apart, k = t)
            constexpr uint32_t id_c = umma::idesc_bf16(128, 128, 1, 1, 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma::mma(tmem + TM_S, umma::sdesc4(sb4 + ((R_DO + b * 16384 + ks * 2048) >> 4), 8192, 1024),
                          umma::sdesc4(sb4 + ((bb + kBlobQT + ks * 2048) >> 4), 8192, 1024), id_c, 1u);
            if (save) {
                umma::bulk_store(P.save_ds + ((size_t)(sbase + j) * H + h) * TILE_S, sb + R_ST, TILE_S);
                umma::bulk_commit();
            }
        }
        if (!umma::mbar_wait(bar_u, pm, WAIT_LIMIT)) {
            timed_out = true;
            pend_m = 0;
            pend_mph = pm;
        }
        umma::fence_after();

        // ------------------------------------------------------------ dU'^T (bf16) operand
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
                *reinterpret_cast<uint4 *>(sm + R_UT + umma::kmaj(jrow, 16 * cg + c, 128)) = pk;
            }
        }
        umma::fence_proxy_async();
        umma::fence_before();
        if (__syncthreads_or(timed_out)) {
            timed_out = true;
            break;
        }

        // ------------------------------------------------------------ dS'^T -= dU'^T W
        if (tid == 0) {
            umma::fence_after();
            // B = W read as K-major (n = key channel i, k = t), negated
            constexpr uint32_t id_d = umma::idesc_bf16(128, 128, 0, 0, 1);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma::mma(tmem + TM_S, umma::sdesc4(sb4 + ((R_UT + ks * 32) >> 4), 16, 1024),
                          umma::sdesc4(sb4 + ((bb + kBlobW + ks * 32) >> 4), 16, 1024), id_d, 1u);
            if (save) {
                // the copies of this chunk's tiles have read them before the
                // products complete, so the next chunk may overwrite them
                umma::bulk_store(P.save_du + ((size_t)(sbase + j) * H + h) * TILE_U, sb + R_UT, TILE_U);
                umma::bulk_commit();
                umma::bulk_wait_read();
            }
            umma::commit(bar_o);
        }
        if (!umma::mbar_wait(bar_o, pm, WAIT_LIMIT)) {
            timed_out = true;
            pend_m = 1;
            pend_mph = pm;
        }
        umma::fence_after();
    }

    if (timed_out) {
        if (tid == 0) report_status(P.status, KDA_STATUS_TIMEOUT);
        // let a copy still in flight land and products still running finish
        // before the shared and tensor memory are released
        if (pend_b >= 0) umma::mbar_wait(bar0 + 8 * pend_b, pend_ph, WAIT_LIMIT);
        if (pend_m >= 0) umma::mbar_wait(pend_m ? bar_o : bar_u, pend_mph, WAIT_LIMIT);
    } else if (cut_out || (segs && P.r_out)) {  // raw dS' to the next piece, or the segment's
        float r[32];
        umma::ld32(tq + TM_S + 32 * cg, r);
        float *dst = cut_out ? P.carry_out + (size_t)h * D * D : P.r_out + uoff;
#pragma unroll
        for (int c = 0; c < 32; ++c) dst[(size_t)(32 * cg + c) * D + jrow] = r[c];
    } else if (P.dS0 && !segs) {
        float r[32];
        umma::ld32(tq + TM_S + 32 * cg, r);
#pragma unroll
        for (int c = 0; c < 32; ++c) P.dS0[uoff + (size_t)(32 * cg + c) * D + jrow] = r[c] * wscale;
    }
    if (save && tid == 0) umma::bulk_wait_all();
    umma::fence_before();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(tmem, 256);
}

// ============================================================================ chunk gradients
// 512 threads: thread (lane l = 32 (warp % 4) + lane, group cg = warp / 4)
// owns TMEM lane l (a key channel, value column or row of the products) and
// the columns of token block cg (tokens 16 cg .. 16 cg + 15), so every per-token
// loop is 16 long and the block anchoring of a channel is thread-local.
constexpr int NB = 512;
// shared memory, 1024-aligned regions.  Phases A and B (the first two
// product batches):
constexpr uint32_t B_SB = 0;        // S^T bf16 [j][i] (K-major 128 x 128)
constexpr uint32_t B_DS = 32768;    // dS'^T bf16 [j][i]
constexpr uint32_t B_DO = 65536;    // dO K-major 64 rows x 128 (rows 0-63 of each 16 KB K block, by TMA)
constexpr uint32_t B_VR = 98304;    // Vres^T bf16 [j][s]
constexpr uint32_t B_UB = 114688;   // U^T bf16 [j][t]   (B_VR + 16 KB: second M block of [Vres; U])
constexpr uint32_t B_DU = 131072;   // dU'^T bf16 [j][t]
constexpr uint32_t B_TBL = 147456;  // the low bf16 part of T diag(b)
constexpr uint32_t B_TN = 155648;   // T bf16, MN-major (n = b, k = t)
constexpr uint32_t B_PT = B_TBL;    // after the first batch: P^T = (T^T dU')^T bf16 [j][a] (16 KB)
constexpr uint32_t B_KT = 163840;   // K~, MN-major (n = t, k = i); then -dVres^T bf16 [j][s]
constexpr uint32_t B_NDV = B_KT;
constexpr uint32_t B_TB = 180224;   // T diag(b), MN-major (n = s, k = t)
constexpr uint32_t B_TF = 188416;   // T f32 [64][64]
constexpr uint32_t B_MT = 204800;   // M^T f32 [64][64]
// the item's rows, staged by TMA where tiles arrive later or are built later:
// k and q [64 t][128] bf16 over U^T and Vres^T, g [64 t][128] f32 over dS'^T
// (those two tiles are copied once the rows are read), v in the rows 64-127
// of the dO tile's K blocks (two 8 KB value halves)
constexpr uint32_t B_KST = B_UB, B_QST = B_VR, B_GST = B_DS;
// phases C and D, over the phase A / B regions once the second batch is done:
constexpr uint32_t B_AP = 0;        // A' K-major 128 rows x 192 (three K blocks of 16 KB)
constexpr uint32_t B_LT0 = 98304;   // L^T K-major 128 channels x 128: K block 0 (k x)
constexpr uint32_t B_RS = 122880;   // R_seg^T K-major 128 channels x 192 (three K blocks)
constexpr uint32_t B_LT1 = 172032;  //   and K block 1 (q x)
constexpr uint32_t B_CUM = B_KT;    // the combine's block sums f32 [8][128] (K~ is built after the
                                    // next item's copies, which go out during the combine, have landed)
constexpr uint32_t B_MISC = 221184;
constexpr uint32_t B_BETA = B_MISC;           // f32 [64]
constexpr uint32_t B_PART = B_MISC + 256;     // f32 [4][128] block decays
constexpr uint32_t B_DGC = B_PART + 2048;     // f32 [8][128] parts of rowsum(dS' . S)
constexpr uint32_t B_DBP = B_DGC + 4096;      // f32 [8][64] beta gradient parts
constexpr uint32_t B_BAR = B_DBP + 2048;      // 5 mbarriers: loads, three product batches, late loads
constexpr uint32_t B_TMEM = B_BAR + 56;
constexpr uint32_t B_CLAIM = B_TMEM + 8;      // int [2]: item in hand, next item
constexpr uint32_t B_SMEM = B_CLAIM + 8 + 1024;
static_assert(B_LT0 + 16384 <= B_RS && B_RS + 49152 <= B_LT1 && B_LT1 + 16384 <= B_TF,
              "phase C regions overlap one another or the kept T and M");
static_assert(B_TN + 8192 <= B_KT, "T tile");
static_assert(B_SMEM <= 232448, "shared memory");
// tensor-memory columns of the products
constexpr uint32_t T1 = 0, T2 = 64, TP = 128, T3 = 0, T4 = 320, T5 = 448, T7 = 192, T8 = 0, T9 = 128;

struct BchunkParams {
    const void *k, *q, *v;           // bf16 [T][H][128]
    const float *g, *beta;           // [T][H][128], [T][H]
    int H;
    float scale, wscale, g_min;
    int zero_do;
    const int2 *list;                // slot -> {first token, length}
    int slot0;                       // first slot of this launch (a piece)
    int nitems;                      // slots x H of this launch; item w (slot0 H + w overall) = slot, head
    int *claim;                      // item counter, zero at launch
    const unsigned char *save_s, *save_u, *save_ds, *save_du;  // [slot][H] tiles
    const float *aux;                // [slot][H][2][64][64]: T, M^T
    CUtensorMap tdo, tv;             // dout, v: box 64 x 1 x 64, 128-byte swizzle
    CUtensorMap tk, tq, tg;          // k, q, g: box 128 x 1 x 64, no swizzle
    float *dq, *dk, *dv, *dg, *dbeta;
    uint32_t *status;
};

__device__ __forceinline__ void sts_bf16x8(uint32_t addr, const float (&v)[8], int o) {
    sts128(addr, pack_bf16(v[o], v[o + 1]), pack_bf16(v[o + 2], v[o + 3]), pack_bf16(v[o + 4], v[o + 5]),
           pack_bf16(v[o + 6], v[o + 7]));
}
__device__ __forceinline__ void sts_bf16x8(uint32_t addr, const float (&v)[16], int o) {
    sts128(addr, pack_bf16(v[o], v[o + 1]), pack_bf16(v[o + 2], v[o + 3]), pack_bf16(v[o + 4], v[o + 5]),
           pack_bf16(v[o + 6], v[o + 7]));
}

__global__ void __launch_bounds__(NB, 1) kda_bwd_chunk_kernel(const __grid_constant__ BchunkParams p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(sm);
    const uint32_t sb4 = sb >> 4;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int qd = warp & 3, cg = warp >> 2;
    const int l = 32 * qd + lane;  // TMEM lane: channel / value column / row owned
    const int c0 = 16 * cg;        // first token (column) of this thread's block
    const int H = p.H;
    float *sBeta = reinterpret_cast<float *>(sm + B_BETA);
    float *sPart = reinterpret_cast<float *>(sm + B_PART);
    float *sDgc = reinterpret_cast<float *>(sm + B_DGC);
    float *sDbp = reinterpret_cast<float *>(sm + B_DBP);
    float *sCum = reinterpret_cast<float *>(sm + B_CUM);
    const float *sTF = reinterpret_cast<const float *>(sm + B_TF);
    const float *sMT = reinterpret_cast<const float *>(sm + B_MT);
    int *sClaim = reinterpret_cast<int *>(sm + B_CLAIM);
    const uint32_t bar = sb + B_BAR;  // bar + 8 k: k = 0 loads, 1..3 product batches, 4 late loads
    const float scale = p.scale, wscale = p.wscale, g_min = p.g_min;

    if (tid == 0) {
        for (int b = 0; b < 5; ++b) umma::mbar_init(bar + 8 * b, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        sClaim[0] = atomicAdd(p.claim, 1);
        sClaim[1] = atomicAdd(p.claim, 1);
    }
    if (warp == 0) umma::tmem_alloc(sb + B_TMEM, 512);
    umma::fence_before();
    __syncthreads();
    umma::fence_after();
    const uint32_t tmem = *reinterpret_cast<const uint32_t *>(sm + B_TMEM);
    const uint32_t tq = tmem + ((uint32_t)(32 * qd) << 16);
    int w = sClaim[0], wn = sClaim[1];
    uint32_t it = 0;
    bool alive = true;
    __syncthreads();  // claims read before thread 0 writes the next ones
    // thread 0 issues an item's copies, all on the loads barrier: the tiles
    // S^T, dU'^T, T | M^T, and the rows (dO and v by swizzled boxes, k, q, g
    // plain).  An item's copies go out during the previous item's combine
    // (every region they fill is free by then) unless that item was skipped.
    auto issue_loads = [&](int wi, int hi, int ti) {
        umma::fence_proxy_async();
        umma::mbar_expect_tx(bar, TILE_S + TILE_U + 4 * AUX_FLOATS + 4 * 16384u + 32768u);
        const size_t wa = (size_t)p.slot0 * p.H + wi;  // (slot, head) index over all slots
        umma::bulk_load(sb + B_SB, p.save_s + wa * TILE_S, TILE_S, bar);
        umma::bulk_load(sb + B_DU, p.save_du + wa * TILE_U, TILE_U, bar);
        umma::bulk_load(sb + B_TF, p.aux + wa * AUX_FLOATS, 4 * AUX_FLOATS, bar);
        umma::tma_load_3d(sb + B_DO, &p.tdo, 0, hi, ti, bar);
        umma::tma_load_3d(sb + B_DO + 16384, &p.tdo, 64, hi, ti, bar);
        umma::tma_load_3d(sb + B_DO + 8192, &p.tv, 0, hi, ti, bar);
        umma::tma_load_3d(sb + B_DO + 24576, &p.tv, 64, hi, ti, bar);
        umma::tma_load_3d(sb + B_KST, &p.tk, 0, hi, ti, bar);
        umma::tma_load_3d(sb + B_QST, &p.tq, 0, hi, ti, bar);
        umma::tma_load_3d(sb + B_GST, &p.tg, 0, hi, ti, bar);
    };
    bool preloaded = false;  // thread 0: the item in hand's copies went out during the previous one
    int2 ncl = make_int2(0, 0);  // thread 0: chunk entry of the next item

    while (w < p.nitems) {
    const int slot = p.slot0 + w / H, h = w % H;
    const size_t wa = (size_t)p.slot0 * H + w;  // (slot, head) index over all slots
    const int2 cl = p.list[slot];
    const int tc = cl.x, Lc = cl.y;
    const uint32_t par = it & 1u;
    if (Lc > 0) {
    uint32_t pend = 0;  // barriers whose wait gave up
    // ---------------------------------------------------------------- loads
    if (tid == 0) {
        if (!preloaded) issue_loads(w, h, tc);
    }
    // thread (channel ch = l, block cg): e^{g} of the block's tokens and their
    // (k, q) as a bf16 pair; x (running product from the block start,
    // inclusive) and y (to the block end, exclusive) are formed where needed
    const int ch = l;
    float e[16];
    uint32_t kq[16];
    uint32_t below = 0;  // bit u: g < g_min (no gradient)
    pend |= umma::mbar_wait(bar, par, it == 0 ? FIRST_WAIT_LIMIT : WAIT_LIMIT) ? 0u : 1u;
#pragma unroll
    for (int u = 0; u < 16; ++u) {
        const int t = c0 + u;
        const bool ok = t < Lc;
        const float gv = ok ? *reinterpret_cast<const float *>(sm + B_GST + t * 512 + ch * 4) : 0.f;
        below |= (ok && gv < g_min) ? (1u << u) : 0u;
        e[u] = __expf(fmaxf(gv, g_min));
        const uint32_t kb = ok ? (uint32_t)lds16(sb + B_KST + t * 256 + ch * 2) : 0u;
        const uint32_t qb = ok ? (uint32_t)lds16(sb + B_QST + t * 256 + ch * 2) : 0u;
        kq[u] = kb | (qb << 16);
    }
    auto prefix = [&](float (&x)[16]) {
        x[0] = e[0];
#pragma unroll
        for (int u = 1; u < 16; ++u) x[u] = x[u - 1] * e[u];
    };
    auto suffix = [&](float (&y)[16]) {
        y[15] = 1.f;
#pragma unroll
        for (int u = 14; u >= 0; --u) y[u] = y[u + 1] * e[u + 1];
    };
    auto kf = [&](int u) { return __uint_as_float(kq[u] << 16); };
    auto qf = [&](int u) { return __uint_as_float(kq[u] & 0xFFFF0000u); };
    {
        float x[16];
        prefix(x);
        sPart[cg * 128 + ch] = x[15];
    }
    if (tid < CH) sBeta[tid] = (tid < Lc) ? p.beta[(size_t)(tc + tid) * H + h] : 0.f;
    __syncthreads();
    float dl[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) dl[m] = sPart[m * 128 + ch];
    // products of the block decays before / after this thread's block
    float pre = 1.f, post = 1.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        if (m < cg) pre *= dl[m];
        if (m > cg) post *= dl[m];
    }
    {  // K~ = K Gam as the MN-major B operand of (K~ S)^T (n = t, k = i = ch)
        float x[16], v[16];
        prefix(x);
#pragma unroll
        for (int u = 0; u < 16; ++u) v[u] = kf(u) * (pre * x[u]);
        sts_bf16x8(sb + B_KT + umma::mnmaj(c0, ch, 1), v, 0);
        sts_bf16x8(sb + B_KT + umma::mnmaj(c0 + 8, ch, 1), v, 8);
    }
    {  // T diag(b) as the MN-major B operand of dVres^T (n = s, k = t), high and low bf16 parts
        const int t = tid >> 3, s = 8 * (tid & 7);
        float tb[8];
#pragma unroll
        for (int e2 = 0; e2 < 8; ++e2) tb[e2] = sTF[t * 64 + s + e2] * sBeta[s + e2];
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e2 = 0; e2 < 8; e2 += 2) {
            hi[e2 >> 1] = pack_bf16(tb[e2], tb[e2 + 1]);
            const float2 h2 = unpack_bf16(hi[e2 >> 1]);
            lo[e2 >> 1] = pack_bf16(tb[e2] - h2.x, tb[e2 + 1] - h2.y);
        }
        sts128(sb + B_TB + umma::mnmaj(s, t, 1), hi[0], hi[1], hi[2], hi[3]);
        sts128(sb + B_TBL + umma::mnmaj(s, t, 1), lo[0], lo[1], lo[2], lo[3]);
        // and T itself, the B operand of P^T = dU'^T T
        const float4 a0 = *reinterpret_cast<const float4 *>(sTF + t * 64 + s);
        const float4 a1 = *reinterpret_cast<const float4 *>(sTF + t * 64 + s + 4);
        sts128(sb + B_TN + umma::mnmaj(s, t, 1), pack_bf16(a0.x, a0.y), pack_bf16(a0.z, a0.w), pack_bf16(a1.x, a1.y),
               pack_bf16(a1.z, a1.w));
    }
    {  // dO rows past the chunk end (every row when dO enters no product) are zero
        const int z0 = p.zero_do ? 0 : Lc;
        for (int idx = tid; idx < (CH - z0) * 16; idx += NB) {
            const int r = z0 + (idx >> 4), c = idx & 15;
            *reinterpret_cast<uint4 *>(sm + B_DO + (c >> 3) * 16384 + r * 128 + (c & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    umma::fence_proxy_async();
    umma::fence_before();
    __syncthreads();

    // ---------------------------------------------------------------- batch 1: (K~ S)^T, dVres^T / wscale, P^T
    // (dA = -T^T dT T^T with dT = dU Vres^T diag(b) and U = T diag(b) Vres is
    // -(T^T dU) U^T: P = T^T dU' here, P U^T with the second batch)
    if (tid == 0) {
        umma::fence_after();
        // the rows are read: the tiles that go over their staging
        umma::fence_proxy_async();
        umma::mbar_expect_tx(bar + 32, TILE_S + TILE_U);
        umma::bulk_load(sb + B_DS, p.save_ds + wa * TILE_S, TILE_S, bar + 32);
        umma::bulk_load(sb + B_UB, p.save_u + wa * TILE_U, TILE_U, bar + 32);
        constexpr uint32_t id1 = umma::idesc_bf16(128, 64, 0, 1, 0);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            umma::mma(tmem + T1, umma::sdesc4(sb4 + ((B_SB + (ks >> 2) * 16384 + (ks & 3) * 32) >> 4), 16, 1024),
                      umma::sdesc4(sb4 + ((B_KT + ks * 2048) >> 4), 1024, 1024), id1, ks > 0 ? 1u : 0u);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            umma::mma(tmem + T2, umma::sdesc4(sb4 + ((B_DU + (ks & 3) * 32) >> 4), 16, 1024),
                      umma::sdesc4(sb4 + (((ks < 4 ? B_TB : B_TBL) + (ks & 3) * 2048) >> 4), 1024, 1024), id1,
                      ks > 0 ? 1u : 0u);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
            umma::mma(tmem + TP, umma::sdesc4(sb4 + ((B_DU + ks * 32) >> 4), 16, 1024),
                      umma::sdesc4(sb4 + ((B_TN + ks * 2048) >> 4), 1024, 1024), id1, ks > 0 ? 1u : 0u);
        umma::commit(bar + 8);
        // the next item's tiles and rows into L2 while this one runs
        ncl = (wn < p.nitems) ? p.list[p.slot0 + wn / H] : make_int2(0, 0);
        if (wn < p.nitems) {
            if (ncl.y > 0) {
                const int hn = wn % H;
                const size_t wna = (size_t)p.slot0 * H + wn;
                umma::prefetch_l2(p.save_s + wna * TILE_S, TILE_S);
                umma::prefetch_l2(p.save_ds + wna * TILE_S, TILE_S);
                umma::prefetch_l2(p.save_u + wna * TILE_U, TILE_U);
                umma::prefetch_l2(p.save_du + wna * TILE_U, TILE_U);
                umma::prefetch_l2(p.aux + wna * AUX_FLOATS, 4 * AUX_FLOATS);
                umma::prefetch_tile_3d(&p.tk, 0, hn, ncl.x);
                umma::prefetch_tile_3d(&p.tq, 0, hn, ncl.x);
                umma::prefetch_tile_3d(&p.tg, 0, hn, ncl.x);
                umma::prefetch_tile_3d(&p.tv, 0, hn, ncl.x);
                umma::prefetch_tile_3d(&p.tv, 64, hn, ncl.x);
                umma::prefetch_tile_3d(&p.tdo, 0, hn, ncl.x);
                umma::prefetch_tile_3d(&p.tdo, 64, hn, ncl.x);
            }
        }
    }
    pend |= umma::mbar_wait(bar + 8, par, WAIT_LIMIT) ? 0u : 2u;
    umma::fence_after();
    {  // thread (value column j = l, block cg): Vres^T and -dVres^T rows j
        const int j = l;
        float a[16];
        umma::ld16(tq + T1 + c0, a);
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int t = c0 + u;
            const float vv =
                (t < Lc) ? __uint_as_float((uint32_t)lds16(sb + B_DO + umma::kmaj(64 + t, j, 128)) << 16) : 0.f;
            a[u] = vv - a[u];
        }
        sts_bf16x8(sb + B_VR + umma::kmaj(j, c0, 128), a, 0);
        sts_bf16x8(sb + B_VR + umma::kmaj(j, c0 + 8, 128), a, 8);
        umma::ld16(tq + T2 + c0, a);
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int s = c0 + u;
            const float dvr = a[u] * wscale;
            if (s < Lc) p.dv[((size_t)(tc + s) * H + h) * D + j] = dvr;
            a[u] = -dvr;
        }
        sts_bf16x8(sb + B_NDV + umma::kmaj(j, c0, 128), a, 0);
        sts_bf16x8(sb + B_NDV + umma::kmaj(j, c0 + 8, 128), a, 8);
        umma::ld16(tq + TP + c0, a);  // P^T row j, columns a = c0 ..
        sts_bf16x8(sb + B_PT + umma::kmaj(j, c0, 128), a, 0);
        sts_bf16x8(sb + B_PT + umma::kmaj(j, c0 + 8, 128), a, 8);
    }
    pend |= umma::mbar_wait(bar + 32, par, WAIT_LIMIT) ? 0u : 16u;
    umma::fence_proxy_async();
    umma::fence_before();
    __syncthreads();

    // ---------------------------------------------------------------- batch 2: Vres dU'^T, dO U^T, S dO^T, -S dVres^T, dS' U^T, P U^T
    if (tid == 0) {
        umma::fence_after();
        constexpr uint32_t id3 = umma::idesc_bf16(128, 64, 1, 1, 0);
        constexpr uint32_t id3b = umma::idesc_bf16(128, 64, 0, 1, 0);
        constexpr uint32_t id4a = umma::idesc_bf16(128, 64, 1, 0, 0);
        constexpr uint32_t id5 = umma::idesc_bf16(128, 64, 1, 1, 0);
        // lanes 0-63: (dU' Vres^T)^T, lane s (A = [Vres; U], rows 64-127 unused)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            umma::mma(tmem + T3, umma::sdesc4(sb4 + ((B_VR + ks * 2048) >> 4), 16384, 1024),
                      umma::sdesc4(sb4 + ((B_DU + ks * 2048) >> 4), 1024, 1024), id3, ks > 0 ? 1u : 0u);
        // lanes 64-127: dO U^T, lane t: A = the K-major dO tile read from 64 rows
        // before it, so its rows 0-63 land in lanes 64-127 (rows 0-63 unused)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            umma::mma(tmem + T3 + 64, umma::sdesc4(sb4 + ((B_DO - 8192 + (ks >> 2) * 16384 + (ks & 3) * 32) >> 4), 16, 1024),
                      umma::sdesc4(sb4 + ((B_UB + ks * 2048) >> 4), 1024, 1024), id3b, ks > 0 ? 1u : 0u);
        // S dO^T (columns 0-63) and -S dVres^T (columns 64-127)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            umma::mma(tmem + T4, umma::sdesc4(sb4 + ((B_SB + ks * 2048) >> 4), 16384, 1024),
                      umma::sdesc4(sb4 + ((B_DO + (ks >> 2) * 16384 + (ks & 3) * 32) >> 4), 16, 1024), id4a,
                      ks > 0 ? 1u : 0u);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            umma::mma(tmem + T4 + 64, umma::sdesc4(sb4 + ((B_SB + ks * 2048) >> 4), 16384, 1024),
                      umma::sdesc4(sb4 + ((B_NDV + ks * 2048) >> 4), 1024, 1024), id5, ks > 0 ? 1u : 0u);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            umma::mma(tmem + T5, umma::sdesc4(sb4 + ((B_DS + ks * 2048) >> 4), 16384, 1024),
                      umma::sdesc4(sb4 + ((B_UB + ks * 2048) >> 4), 1024, 1024), id5, ks > 0 ? 1u : 0u);
        // lanes 0-63: P U^T, lane a (A = P^T read MN-major, rows 64-127 unused)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
            umma::mma(tmem + T7, umma::sdesc4(sb4 + ((B_PT + ks * 2048) >> 4), 16384, 1024),
                      umma::sdesc4(sb4 + ((B_UB + ks * 2048) >> 4), 1024, 1024), id3, ks > 0 ? 1u : 0u);
        umma::commit(bar + 16);
    }
    {  // rowsum(dS' . S): key channels 2 cp, 2 cp + 1 over value columns 16 jg .. 16 jg + 15
        const int cp = tid & 63, jg = tid >> 6;
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll 8
        for (int jj = 0; jj < 16; ++jj) {
            const int j = 16 * jg + jj;
            const float2 a = unpack_bf16(lds32(sb + B_DS + umma::kmaj(j, 2 * cp, 128)));
            const float2 b = unpack_bf16(lds32(sb + B_SB + umma::kmaj(j, 2 * cp, 128)));
            acc = __ffma2_rn(a, b, acc);
        }
        *reinterpret_cast<float2 *>(sDgc + jg * 128 + 2 * cp) = acc;
    }
    pend |= umma::mbar_wait(bar + 16, par, WAIT_LIMIT) ? 0u : 4u;
    umma::fence_after();
    __syncthreads();  // every thread is done with the S and dS' tiles
    // the phase A / B regions are free: zero A'; meanwhile the anchored
    // operands of the last batch, which no readout below touches
    for (int idx = tid; idx < 49152 / 16; idx += NB)
        *reinterpret_cast<uint4 *>(sm + B_AP + idx * 16) = make_uint4(0u, 0u, 0u, 0u);
    {  // the anchored column operand R_seg^T: for segment i >= cg,
       // R_i[s] = k_s y_s c_i with c_i = 1 / delta_cg (i = cg), else the decays
       // of the blocks strictly between
        float y[16];
        suffix(y);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (i < cg) continue;
            float c = 1.f;
            if (i == cg) {
                c = __frcp_rn(dl[cg]);
            } else {
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    if (m > cg && m < i) c *= dl[m];
            }
            float a[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) a[u] = kf(u) * (y[u] * c);
            sts_bf16x8(sb + B_RS + umma::kmaj(ch, segoff(i) + c0, 128), a, 0);
            sts_bf16x8(sb + B_RS + umma::kmaj(ch, segoff(i) + c0 + 8, 128), a, 8);
        }
    }
    {  // the anchored row operand L^T (row ch: k x in K block 0, q x in K block 1)
        float x[16], a[16], b[16];
        prefix(x);
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            a[u] = kf(u) * x[u];
            b[u] = qf(u) * x[u];
        }
        sts_bf16x8(sb + B_LT0 + umma::kmaj(ch, c0, 128), a, 0);
        sts_bf16x8(sb + B_LT0 + umma::kmaj(ch, c0 + 8, 128), a, 8);
        sts_bf16x8(sb + B_LT1 + umma::kmaj(ch, c0, 128), b, 0);
        sts_bf16x8(sb + B_LT1 + umma::kmaj(ch, c0 + 8, 128), b, 8);
    }
    __syncthreads();  // A' zeroed before its rows are written
    if (qd < 2) {
        {  // lanes 0-63: s = l; columns t: dTB[t][s] / wscale -> beta gradient
            const int s = l;
            float a[16];
            umma::ld16(tq + T3 + c0, a);
            float dbp = 0.f;
#pragma unroll
            for (int u = 0; u < 16; ++u) dbp = fmaf(a[u] * wscale, sTF[(c0 + u) * 64 + s], dbp);
            sDbp[cg * 64 + s] = dbp;
        }
        {  // row a = l of dA = -wscale P U^T (strictly lower): beta gradient, dM into A' row a
            const int a = l, ba_blk = a >> 4;
            float v[16];
            umma::ld16(tq + T7 + c0, v);
            const float ba = sBeta[a];
            float dbp = 0.f;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int b = c0 + u;
                const float da = (b < a) ? -wscale * v[u] : 0.f;
                dbp = fmaf(da, sMT[b * 64 + a], dbp);
                v[u] = ba * da;
            }
            sDbp[256 + cg * 64 + a] = dbp;
            if (cg <= ba_blk) {
                sts_bf16x8(sb + B_AP + umma::kmaj(a, segoff(ba_blk) + c0, 128), v, 0);
                sts_bf16x8(sb + B_AP + umma::kmaj(a, segoff(ba_blk) + c0 + 8, 128), v, 8);
            }
        }
    } else {  // lanes 64-127: t = l - 64; columns 64 + s: (dO U^T)[t][s] -> A' row 64 + t (s <= t)
        const int t = l - 64, bt = t >> 4;
        float a[16];
        umma::ld16(tq + T3 + 64 + c0, a);
        if (cg <= bt) {  // the columns of this block lie in the segment of row t
#pragma unroll
            for (int u = 0; u < 16; ++u) a[u] = (c0 + u <= t) ? scale * a[u] : 0.f;
            sts_bf16x8(sb + B_AP + umma::kmaj(64 + t, segoff(bt) + c0, 128), a, 0);
            sts_bf16x8(sb + B_AP + umma::kmaj(64 + t, segoff(bt) + c0 + 8, 128), a, 8);
        }
    }
    umma::fence_proxy_async();
    umma::fence_before();
    __syncthreads();

    // ---------------------------------------------------------------- batch 3: dL = A' R_seg, dR_seg = A'^T L
    if (tid == 0) {
        umma::fence_after();
        constexpr uint32_t id8 = umma::idesc_bf16(128, 128, 0, 0, 0);
        constexpr uint32_t id9 = umma::idesc_bf16(128, 160, 0, 1, 0);
#pragma unroll
        for (int ks = 0; ks < 10; ++ks) {
            const uint32_t kb = ks >> 2, kin = (ks & 3) * 32;
            umma::mma(tmem + T8, umma::sdesc4(sb4 + ((B_RS + kb * 16384 + kin) >> 4), 16, 1024),
                      umma::sdesc4(sb4 + ((B_AP + kb * 16384 + kin) >> 4), 16, 1024), id8, ks > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint32_t kb = ks >> 2, kin = (ks & 3) * 32;
            umma::mma(tmem + T9, umma::sdesc4(sb4 + (((kb ? B_LT1 : B_LT0) + kin) >> 4), 16, 1024),
                      umma::sdesc4(sb4 + ((B_AP + ks * 2048) >> 4), 16384, 1024), id9, ks > 0 ? 1u : 0u);
        }
        umma::commit(bar + 24);
    }
    if (tid < CH && tid < Lc) {
        float db = 0.f;
#pragma unroll
        for (int pq = 0; pq < 8; ++pq) db += sDbp[pq * 64 + tid];
        p.dbeta[(size_t)(tc + tid) * H + h] = db;
    }
    pend |= umma::mbar_wait(bar + 24, par, WAIT_LIMIT) ? 0u : 8u;
    umma::fence_after();
    if (tid == 0) {  // every product has read its operands: the next item's copies, and the one after claimed
        preloaded = wn < p.nitems && ncl.y > 0 && pend == 0;
        if (preloaded) issue_loads(wn, wn % H, ncl.x);
        sClaim[0] = (wn < p.nitems) ? atomicAdd(p.claim, 1) : p.nitems;
    }

    // ---------------------------------------------------------------- token gradients of channel ch, block cg
    {
        const float gamC = dl[0] * dl[1] * dl[2] * dl[3];
        float dsum = 0.f;
#pragma unroll
        for (int jg = 0; jg < 8; ++jg) dsum += sDgc[jg * 128 + ch];
        const float dgc = gamC * wscale * dsum;
        float dgam[16];
        float2 sh2 = make_float2(0.f, 0.f);  // sum over this block of dK^ . K^ (even, odd tokens)
        // column factors of the segments i >= cg (see R_seg^T)
        float cs[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float c = 1.f;
            if (i == cg) {
                c = __frcp_rn(dl[cg]);
            } else {
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    if (m > cg && m < i) c *= dl[m];
            }
            cs[i] = c;
        }
        float xr = 1.f, y[16];
        suffix(y);
#pragma unroll
        for (int u0 = 0; u0 < 16; u0 += 4) {
            const int t0 = c0 + u0;
            // every column group of these 4 tokens in one round of loads
            uint32_t a4[4], a5[4], a6[4], a7[4], a8[4], r9[4][4];
            umma::ld4_async(tq + T4 + t0, a4);       // S dO^T
            umma::ld4_async(tq + T4 + 64 + t0, a5);  // -S dVres^T
            umma::ld4_async(tq + T5 + t0, a6);       // dS' U^T
            umma::ld4_async(tq + T8 + t0, a7);       // dL (k rows)
            umma::ld4_async(tq + T8 + 64 + t0, a8);  // dL (q rows)
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (i >= cg) umma::ld4_async(tq + T9 + segoff(i) + t0, r9[i]);  // dR_seg
            umma::wait_ld();
            umma::hold(a4);
            umma::hold(a5);
            umma::hold(a6);
            umma::hold(a7);
            umma::hold(a8);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (i >= cg) umma::hold(r9[i]);
            // two tokens at a time as packed f32x2 operations (each lane rounds
            // like the scalar operation)
#pragma unroll
            for (int pr = 0; pr < 4; pr += 2) {
                const int u = u0 + pr, t = t0 + pr;
                const float x0 = xr * e[u], x1 = x0 * e[u + 1];  // x of the two tokens
                xr = x1;
                const float2 xx = make_float2(x0, x1), yy = make_float2(y[u], y[u + 1]);
                const float2 kk = make_float2(kf(u), kf(u + 1)), qq = make_float2(qf(u), qf(u + 1));
                float2 kc = make_float2(0.f, 0.f), rr = kc;  // sum_i f_i dR_i, sum_i R_i dR_i (R_i as the product read it)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if (i < cg) continue;
                    const float2 f = __fmul2_rn(yy, make_float2(cs[i], cs[i]));
                    const float2 r = make_float2(__uint_as_float(r9[i][pr]), __uint_as_float(r9[i][pr + 1]));
                    kc = __ffma2_rn(f, r, kc);
                    const float2 kf2 = __fmul2_rn(kk, f);
                    rr = __ffma2_rn(__bfloat1622float2(__floats2bfloat162_rn(kf2.x, kf2.y)), r, rr);
                }
                const float2 gam = __fmul2_rn(make_float2(pre, pre), xx), suf = __fmul2_rn(yy, make_float2(post, post));
                const float2 v4 = make_float2(__uint_as_float(a4[pr]), __uint_as_float(a4[pr + 1]));
                const float2 v5 = make_float2(__uint_as_float(a5[pr]), __uint_as_float(a5[pr + 1]));
                const float2 v6 = make_float2(__uint_as_float(a6[pr]), __uint_as_float(a6[pr + 1]));
                const float2 v7 = make_float2(__uint_as_float(a7[pr]), __uint_as_float(a7[pr + 1]));
                const float2 v8 = make_float2(__uint_as_float(a8[pr]), __uint_as_float(a8[pr + 1]));
                const float2 dqs = __fmul2_rn(make_float2(scale, scale), v4);
                const float2 dq = __ffma2_rn(dqs, gam, __fmul2_rn(xx, v8));
                const float2 kh = __fmul2_rn(__fmul2_rn(make_float2(wscale, wscale), v6), suf);
                const float2 dk = __fadd2_rn(__fadd2_rn(__ffma2_rn(v5, gam, __fmul2_rn(xx, v7)), kc), kh);
                // the anchored terms with the bf16 values of L and R_seg that the
                // products used: each (row, column) pair inside [t, 63] then
                // cancels in the reverse cumulative sum as it does exactly
                const float2 lk = __fmul2_rn(kk, xx), lq = __fmul2_rn(qq, xx);
                const float2 lkb = __bfloat1622float2(__floats2bfloat162_rn(lk.x, lk.y));
                const float2 lqb = __bfloat1622float2(__floats2bfloat162_rn(lq.x, lq.y));
                float2 dg = __ffma2_rn(dqs, __fmul2_rn(qq, gam), __fmul2_rn(v5, __fmul2_rn(kk, gam)));
                dg = __ffma2_rn(make_float2(-kh.x, -kh.y), kk, dg);
                dg = __fadd2_rn(dg, __ffma2_rn(lkb, v7, __fmul2_rn(lqb, v8)));
                dg = __fadd2_rn(dg, make_float2(-rr.x, -rr.y));
                dgam[u] = dg.x;
                dgam[u + 1] = dg.y;
                sh2 = __ffma2_rn(kh, kk, sh2);
                if (t < Lc) {
                    const size_t o = ((size_t)(tc + t) * H + h) * D + ch;
                    p.dq[o] = dq.x;
                    p.dk[o] = dk.x;
                }
                if (t + 1 < Lc) {
                    const size_t o = ((size_t)(tc + t + 1) * H + h) * D + ch;
                    p.dq[o] = dq.y;
                    p.dk[o] = dk.y;
                }
            }
        }
        float tot = 0.f;
#pragma unroll
        for (int u = 0; u < 16; ++u) tot += dgam[u];
        sCum[cg * 128 + ch] = tot;
        sCum[(4 + cg) * 128 + ch] = sh2.x + sh2.y;
        __syncthreads();
        // gamma_C (and the K^ factors through it) collects at the chunk's last
        // token, so it adds to the reverse cumulative sum at every token
        float acc = dgc + ((sCum[512 + ch] + sCum[640 + ch]) + (sCum[768 + ch] + sCum[896 + ch]));
#pragma unroll
        for (int c = 3; c > 0; --c)
            if (c > cg) acc += sCum[c * 128 + ch];
#pragma unroll
        for (int u = 15; u >= 0; --u) {
            acc += dgam[u];
            const int t = c0 + u;
            if (t < Lc) p.dg[((size_t)(tc + t) * H + h) * D + ch] = ((below >> u) & 1u) ? 0.f : acc;
        }
    }
    umma::fence_before();
    ++it;
    if (__syncthreads_or(pend != 0)) {  // uniform: leave once the copies and products in flight are done
        if (pend & 1u) umma::mbar_wait(bar, par, WAIT_LIMIT);
        for (int b = 1; b < 5; ++b)
            if (pend & (1u << b)) umma::mbar_wait(bar + 8 * b, par, WAIT_LIMIT);
        if (tid == 0 && preloaded) umma::mbar_wait(bar, par ^ 1u, WAIT_LIMIT);  // the next item's copies
        alive = false;
        break;
    }
    } else if (tid == 0) {  // Lc > 0: nothing to do for this item; claim the one after the next
        preloaded = false;
        sClaim[0] = (wn < p.nitems) ? atomicAdd(p.claim, 1) : p.nitems;
    }
    __syncthreads();
    w = wn;
    wn = sClaim[0];
    __syncthreads();  // the claim was read by every thread before thread 0 writes the next
    }  // items
    if (!alive && tid == 0) report_status(p.status, KDA_STATUS_TIMEOUT);
    umma::fence_before();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(tmem, 512);
    // launched as a programmatic dependent of a reverse walk: finish only
    // after that walk has, so the next launch on the stream (which waits for
    // this one) also follows it (a no-op for an ordinary launch)
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

// ============================================================================ reverse composition
// The state gradient over context-parallel segments: with the forward
// transition of segment p, S_end = M_p S_start + N_p, and r_p the raw
// gradient a segment's reverse walk reaches at its start from zero at its
// end, dS'_start = M_p^T dS'_end + r_p (all linear in dS' = dS / scale).  One
// CTA per (sequence, head, 16 value columns) runs a sequence's segments last
// to first in fp32, leaving dS' at every segment's end (the start of each
// segment's second reverse walk) and scale dS' at the sequence start (dS0).
constexpr int NC = 256;
struct BcomposeParams {
    const float *M;        // [P][H][dk][dk] forward transitions
    const float *r;        // [P][H][dk][dv] raw dS' at each segment start, from zero
    const int32_t *first;  // [N + 1] first segment of each sequence
    const int32_t *cu;     // [N + 1] sequence bounds (an empty sequence passes dS_final through)
    const float *dS_final; // [N][H][dk][dv] or null (zero)
    float *dS_end;         // [P][H][dk][dv] raw dS' at each segment end
    float *dS0;            // [N][H][dk][dv] or null
    int H;
    float wscale;
};

__global__ void __launch_bounds__(NC) kda_bwd_compose_kernel(const __grid_constant__ BcomposeParams P) {
    __shared__ float cur[D][17];  // raw dS' of this CTA's 16 value columns
    const int n = blockIdx.x, h = blockIdx.y, c0 = 16 * blockIdx.z, tid = threadIdx.x;
    const int H = P.H, pf = P.first[n], pl = P.first[n + 1];
    const float inv = 1.0f / P.wscale;
    if (P.cu[n] == P.cu[n + 1]) {
        if (P.dS0)
            for (int e = tid; e < D * 16; e += NC) {
                const size_t o = (((size_t)n * H + h) * D + (e >> 4)) * D + c0 + (e & 15);
                P.dS0[o] = P.dS_final ? P.dS_final[o] : 0.f;
            }
        return;
    }
    for (int e = tid; e < D * 16; e += NC) {
        const int i = e >> 4, c = e & 15;
        cur[i][c] = P.dS_final ? P.dS_final[(((size_t)n * H + h) * D + i) * D + c0 + c] * inv : 0.f;
    }
    __syncthreads();
    // thread (key row i, 8 columns): out[i][c] = sum_k M_p[k][i] cur[k][c] + r_p[i][c]
    const int i = tid & (D - 1), cq = 8 * (tid >> 7);
    for (int pp = pl - 1; pp >= pf; --pp) {
        const size_t so = ((size_t)pp * H + h) * D * D;
        float acc[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            P.dS_end[so + (size_t)i * D + c0 + cq + c] = cur[i][cq + c];
            acc[c] = P.r[so + (size_t)i * D + c0 + cq + c];
        }
        const float *Mp = P.M + so;
#pragma unroll 4
        for (int k = 0; k < D; ++k) {
            const float m = Mp[(size_t)k * D + i];
#pragma unroll
            for (int c = 0; c < 8; ++c) acc[c] = fmaf(m, cur[k][cq + c], acc[c]);
        }
        __syncthreads();  // every thread has read cur
#pragma unroll
        for (int c = 0; c < 8; ++c) cur[i][cq + c] = acc[c];
        __syncthreads();
    }
    if (P.dS0) {
#pragma unroll
        for (int c = 0; c < 8; ++c)
            P.dS0[(((size_t)n * H + h) * D + i) * D + c0 + cq + c] = cur[i][cq + c] * P.wscale;
    }
}

}  // namespace bt

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
// dout (or v) [T][H][128] bf16, box 64 x 1 head x 64 tokens, 128-byte swizzle
bool encode_dout(CUtensorMap *m, const void *dout, int T, int H) {
    if (T <= 0) return true;  // no chunk: the map is never used
    EncodeTiledFn fn = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
    if (!fn) return false;
    cuuint64_t dims[3] = {128u, (cuuint64_t)H, (cuuint64_t)(T > 0 ? T : 1)};
    cuuint64_t strides[2] = {256u, 256u * (cuuint64_t)H};
    cuuint32_t box[3] = {64u, 1u, 64u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(dout), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// [T][H][128] rows, box 128 x 1 head x 64 tokens, no swizzle
bool encode_plain(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize, int T, int H) {
    if (T <= 0) return true;
    EncodeTiledFn fn = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
    if (!fn) return false;
    cuuint64_t dims[3] = {128u, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {128u * (cuuint64_t)esize, 128u * (cuuint64_t)esize * H};
    cuuint32_t box[3] = {128u, 1u, 64u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    return fn(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

cudaError_t launch_bwd_walk(const BwdTcArgs &a, int slot0, int slot1, const float *carry_in, float *carry_out,
                            cudaStream_t st, const BwdSegments *sg) {
    if (a.N <= 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(bt::kda_bwd_walk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         bt::R_SMEM);
    if (e != cudaSuccess) return e;
    bt::RwalkParams P;
    memset(&P, 0, sizeof(P));
    P.cu = a.cu_seqlens;
    P.N = a.N;
    P.T = a.T;
    P.H = a.H;
    if (!encode_dout(&P.tdo, a.dout, a.T, a.H)) return cudaErrorInvalidValue;
    P.blob = a.blob;
    P.dS_final = a.dS_final;
    P.dS0 = a.dS0;
    P.zero_do = a.scale == 0.f ? 1 : 0;
    P.wscale = a.scale == 0.f ? 1.f : a.scale;
    P.save_ds = a.save_ds;
    P.save_du = a.save_du;
    P.slot0 = slot0;
    P.slot1 = slot1;
    P.carry_in = carry_in;
    P.carry_out = carry_out;
    P.status = a.status;
    int units = a.N;
    if (sg) {  // segments: no pieces, no tiles in the first pass
        P.seg_table = sg->table;
        P.seg_count = sg->count;
        P.dS_in = sg->dS_in;
        P.r_out = sg->r_out;
        P.dS0 = nullptr;
        if (!sg->save) P.save_ds = P.save_du = nullptr;
        units = sg->P_max;
    }
    bt::kda_bwd_walk_kernel<<<dim3(units, a.H), bt::NR, bt::R_SMEM, st>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_bwd_compose(const float *M, const float *r, const int32_t *first, const int32_t *cu,
                               const float *dS_final, float *dS_end, float *dS0, int N, int H, float scale,
                               cudaStream_t st) {
    if (N <= 0) return cudaSuccess;
    bt::BcomposeParams P;
    P.M = M;
    P.r = r;
    P.first = first;
    P.cu = cu;
    P.dS_final = dS_final;
    P.dS_end = dS_end;
    P.dS0 = dS0;
    P.H = H;
    P.wscale = scale == 0.f ? 1.f : scale;
    bt::kda_bwd_compose_kernel<<<dim3(N, H, bt::D / 16), bt::NC, 0, st>>>(P);
    return cudaGetLastError();
}

cudaError_t launch_bwd_chunk(const BwdTcArgs &a, int slot0, int slot1, int *claim, bool after_walk,
                             cudaStream_t st) {
    const int nslots = slot1 - slot0;
    if (nslots <= 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(bt::kda_bwd_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         bt::B_SMEM);
    if (e != cudaSuccess) return e;
    bt::BchunkParams P;
    memset(&P, 0, sizeof(P));
    P.k = a.k;
    P.q = a.q;
    P.v = a.v;
    P.g = a.g;
    P.beta = a.beta;
    P.H = a.H;
    P.scale = a.scale;
    P.zero_do = a.scale == 0.f ? 1 : 0;
    P.wscale = a.scale == 0.f ? 1.f : a.scale;
    P.g_min = a.g_min;
    P.list = a.list;
    P.slot0 = slot0;
    P.nitems = nslots * a.H;
    P.claim = claim;
    P.save_s = a.save_s;
    P.save_u = a.save_u;
    P.save_ds = a.save_ds;
    P.save_du = a.save_du;
    P.aux = a.aux;
    if (!encode_dout(&P.tdo, a.dout, a.T, a.H) || !encode_dout(&P.tv, a.v, a.T, a.H) ||
        !encode_plain(&P.tk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T, a.H) ||
        !encode_plain(&P.tq, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.T, a.H) ||
        !encode_plain(&P.tg, a.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.T, a.H))
        return cudaErrorInvalidValue;
    P.dq = a.dq;
    P.dk = a.dk;
    P.dv = a.dv;
    P.dg = a.dg;
    P.dbeta = a.dbeta;
    P.status = a.status;
    static int sms = 0;
    if (sms <= 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            sms <= 0) {
            cudaGetLastError();
            sms = 152;
        }
    }
    const int grid = P.nitems < sms ? P.nitems : sms;  // persistent: one CTA per SM
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(bt::NB);
    cfg.dynamicSmemBytes = bt::B_SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_walk ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, bt::kda_bwd_chunk_kernel, P);
}

}  // namespace kda
