// decode_token.cu -- single-token decode (draft window 0) on the CUDA cores, sm_103a.
//
// "Noyaux d'inference", section 1 "Le decodage KDA", subsection "La fusion":
// one kernel runs short conv -> input norm -> gating -> recurrence -> output
// norm.  With no draft window the request's only token is the bonus token, so
// the replay tile of the verify kernel degenerates to one step of the
// recurrence, done here directly in fp32 (no tensor cores are needed):
//   D   = Diag(e^g) S                       (decay of the key rows)
//   p   = D^T k^,  r = D^T q^               (column sums over dk)
//   u   = b (v - p)
//   S'  = D + k^ u^T                        (= (I - b k^ k^T) Diag(e^g) S + b k^ v^T)
//   o   = scale S'^T q^ = scale (r + u (k^ . q^))  -> RMSNorm over dv
// One CTA of 256 threads per (request, head); thread (cg, rg) owns the 8
// value columns 8 cg .. 8 cg + 7 of rows rg * RPT .. + RPT - 1 of the bf16
// state: 16-byte copies in (through shared memory, started first), 16-byte
// stores out.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace dtk {

constexpr int NT = 256, NW = NT / 32;

template <int D>
__global__ void __launch_bounds__(NT, 5) kda_decode_token_kernel(VerifyArgs p) {
    constexpr int CG = D / 8;     // column groups of 8 bf16 (16 bytes)
    constexpr int RG = NT / CG;   // row groups
    constexpr int RPT = D / RG;   // rows per thread
    constexpr int DW = D / 32;    // warps that hold one channel each
    __shared__ float sQ[D], sK[D], sV[D], sE[D], sUk[D];
    __shared__ float sNorm[3][DW], sNorm2[DW];
    __shared__ float sRed[NW][CG * 16];  // per warp: k^T D and q^T D partial column sums
    __shared__ __align__(16) __nv_bfloat16 sS[D * D];  // the state, row-major [dk][dv]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.H, W = p.W;
    const int unit = blockIdx.x, h = unit % H, r = unit / H;
    if (p.accepted[r] != 0) {  // window 0: the accepted length must be 0
        if (tid == 0 && h == 0) report_status(p.status, KDA_STATUS_BAD_ACCEPTED_LEN);
        return;
    }
    if (p.draft_len && p.draft_len[r] != 0) {  // and so must the draft count
        if (tid == 0 && h == 0) report_status(p.status, KDA_STATUS_BAD_DRAFT_LEN);
        return;
    }

    // ---------------------------------------------------------------- state read (first, to overlap)
    // each thread copies its own 16-byte pieces into shared memory and reads
    // them back after the norms (no cross-thread hand-off)
    const int cg = tid % CG, rg = tid / CG;
    __nv_bfloat16 *stg = reinterpret_cast<__nv_bfloat16 *>(p.state) + ((size_t)r * H + h) * D * D;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const size_t e = (size_t)(rg * RPT + i) * D + 8 * cg;
        cp_async16(sS + e, stg + e, true);
    }
    cp_async_commit();

    // ---------------------------------------------------------------- conv, gates, norms
    const size_t HD = (size_t)H * D, Cq = 3 * HD;
    if (tid < D) {
        const int c = tid;
        const size_t chq = (size_t)h * D + c;
        const uint16_t *tail = reinterpret_cast<const uint16_t *>(p.tail);
        const uint16_t *nq = reinterpret_cast<const uint16_t *>(p.new_qkv) + (size_t)r * Cq;
        // window rows 0 .. W-2 are the conv tail, row W-1 the token
        uint16_t xq[4], xk[4], xv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            xq[j] = xk[j] = xv[j] = 0;
            if (j < W) {
                const uint16_t *row = (j < W - 1) ? tail + ((size_t)r * (W - 1) + j) * Cq : nq;
                xq[j] = row[chq];
                xk[j] = row[HD + chq];
                xv[j] = row[2 * HD + chq];
            }
        }
        float yq = 0.f, yk = 0.f, yv = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (j < W) {
                yq = fmaf(p.conv_w[chq * W + j], __uint_as_float((uint32_t)xq[j] << 16), yq);
                yk = fmaf(p.conv_w[(HD + chq) * W + j], __uint_as_float((uint32_t)xk[j] << 16), yk);
                yv = fmaf(p.conv_w[(2 * HD + chq) * W + j], __uint_as_float((uint32_t)xv[j] << 16), yv);
            }
        }
        if (p.conv_act == KDA_CONV_SILU) {
            yq = yq / (1.f + __expf(-yq));
            yk = yk / (1.f + __expf(-yk));
            yv = yv / (1.f + __expf(-yv));
        }
        // conv tail write-back: tail row m <- window row m + 1 (bitwise), read above
        uint16_t *tw = reinterpret_cast<uint16_t *>(p.tail);
#pragma unroll
        for (int m = 0; m < 3; ++m) {
            if (m < W - 1) {
                uint16_t *row = tw + ((size_t)r * (W - 1) + m) * Cq;
                row[chq] = xq[m + 1];
                row[HD + chq] = xk[m + 1];
                row[2 * HD + chq] = xv[m + 1];
            }
        }
        // decay e^{max(-softplus(g), g_min)} = max(1 / (1 + e^g), e^{g_min})
        const float graw = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p.new_g)[(size_t)r * HD + chq]);
        sE[c] = fmaxf(1.f / (1.f + __expf(graw)), __expf(p.g_min));
        sQ[c] = yq;
        sK[c] = yk;
        sV[c] = yv;
        float a0 = yq * yq, a1 = yk * yk, a2 = yq * yk;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            a0 += __shfl_xor_sync(0xffffffffu, a0, o);
            a1 += __shfl_xor_sync(0xffffffffu, a1, o);
            a2 += __shfl_xor_sync(0xffffffffu, a2, o);
        }
        if (lane == 0) {
            sNorm[0][warp] = a0;
            sNorm[1][warp] = a1;
            sNorm[2][warp] = a2;
        }
    }
    __syncthreads();
    float nq2 = 0.f, nk2 = 0.f, qk = 0.f;
#pragma unroll
    for (int w = 0; w < DW; ++w) {
        nq2 += sNorm[0][w];
        nk2 += sNorm[1][w];
        qk += sNorm[2][w];
    }
    const float rq = rsqrtf(nq2 + p.eps_in), rk = rsqrtf(nk2 + p.eps_in);
    const float kq = qk * rq * rk;  // k^ . q^

    // ---------------------------------------------------------------- column sums of D = Diag(e^g) S
    // (D is recomputed from the shared copy for the write-back)
    cp_async_wait_all();
    float pk[8], pq[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) pk[j] = pq[j] = 0.f;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int row = rg * RPT + i;
        const float e = sE[row], kr = sK[row], qr = sQ[row];
        const uint4 sv = *reinterpret_cast<const uint4 *>(sS + (size_t)row * D + 8 * cg);
        const uint32_t w4[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 f = unpack_bf16(w4[q]);
            const float d0 = e * f.x, d1 = e * f.y;
            pk[2 * q] = fmaf(kr, d0, pk[2 * q]);
            pq[2 * q] = fmaf(qr, d0, pq[2 * q]);
            pk[2 * q + 1] = fmaf(kr, d1, pk[2 * q + 1]);
            pq[2 * q + 1] = fmaf(qr, d1, pq[2 * q + 1]);
        }
    }
    // over the row groups of this warp (lanes with equal cg), then across warps
#pragma unroll
    for (int o = CG; o < 32; o <<= 1) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            pk[j] += __shfl_xor_sync(0xffffffffu, pk[j], o);
            pq[j] += __shfl_xor_sync(0xffffffffu, pq[j], o);
        }
    }
    if (lane < CG) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            sRed[warp][cg * 16 + j] = pk[j];
            sRed[warp][cg * 16 + 8 + j] = pq[j];
        }
    }
    __syncthreads();

    // ---------------------------------------------------------------- u, outputs
    float oj = 0.f;
    if (tid < D) {
        const int j = tid, g8 = j >> 3, jj = j & 7;
        float sk = 0.f, sq = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            sk += sRed[w][g8 * 16 + jj];
            sq += sRed[w][g8 * 16 + 8 + jj];
        }
        float beta;
        {
            const float braw = __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p.new_b)[(size_t)r * H + h]);
            beta = 1.f / (1.f + __expf(-braw));
        }
        const float u = beta * (sV[j] - rk * sk);
        sUk[j] = rk * u;  // S' = D + k u^T with k = rk * y_k
        oj = p.scale * (rq * sq + u * kq);
        float s2 = oj * oj;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
        if (lane == 0) sNorm2[warp] = s2;
    }
    __syncthreads();

    // ---------------------------------------------------------------- write-back, output
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int row = rg * RPT + i;
        const float e = sE[row], kr = sK[row];
        const uint4 sv = *reinterpret_cast<const uint4 *>(sS + (size_t)row * D + 8 * cg);
        const uint32_t s4[4] = {sv.x, sv.y, sv.z, sv.w};
        uint32_t w4[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 f = unpack_bf16(s4[q]);
            w4[q] = pack_bf16(fmaf(kr, sUk[8 * cg + 2 * q], e * f.x), fmaf(kr, sUk[8 * cg + 2 * q + 1], e * f.y));
        }
        *reinterpret_cast<uint4 *>(stg + (size_t)row * D + 8 * cg) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
    }
    if (tid < D) {
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < DW; ++w) tot += sNorm2[w];
        const float rs = rsqrtf(tot / D + p.eps_out);
        reinterpret_cast<__nv_bfloat16 *>(p.o)[((size_t)r * H + h) * D + tid] =
            __float2bfloat16_rn(oj * rs * p.out_w[tid]);
    }
}

template <int D>
static cudaError_t launch_t(const VerifyArgs &a, cudaStream_t st) {
    const size_t units = (size_t)a.R * a.H;
    kda_decode_token_kernel<D><<<(unsigned)units, NT, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace dtk

cudaError_t launch_decode_token(const VerifyArgs &a, cudaStream_t st) {
    if (a.R <= 0) return cudaSuccess;
    if (a.Wd != 0 || a.dk != a.dv) return cudaErrorInvalidValue;
    if (a.dk == 128) return dtk::launch_t<128>(a, st);
    if (a.dk == 64) return dtk::launch_t<64>(a, st);
    return cudaErrorInvalidValue;
}

}  // namespace kda
