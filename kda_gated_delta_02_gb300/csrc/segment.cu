// segment.cu -- ordered composition of segment transitions on sm_103a.
//
// "Noyaux KDA et FlashKDA", section "Le parallelisme de contexte
// intra-appareil": each segment's transition S -> M S + N is evaluated without
// its incoming state and merged afterwards to recover every segment's exact
// initial state; "Dentro de los esfuerzos de optimizacion de Kimi K3",
// section 5: an ordered scan of the group summaries.
//
// Columns of S are independent under S -> M S + N, so one CTA owns a 16-column
// strip of one (chain, head) and walks the chain's segments in order: stage
// M_p in shared memory (coalesced 16-byte copies), then S <- M_p S + N_p in
// fp32 on the CUDA cores.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

constexpr int CMP_THREADS = 256;
constexpr int STRIP = 16;

template <int DK>
struct ComposeSmem {
    static constexpr int LDM = DK + 4;
    static constexpr int off_m = 0;
    static constexpr int off_s = off_m + DK * LDM * 4;
    static constexpr int bytes = off_s + DK * STRIP * 4;
};

template <int DK>
__global__ void __launch_bounds__(CMP_THREADS) kda_compose_kernel(ComposeArgs a) {
    using L = ComposeSmem<DK>;
    constexpr int LDM = L::LDM;
    constexpr int CPT = DK * STRIP / CMP_THREADS;  // outputs per thread (8 or 4)
    constexpr int GROUPS = STRIP / CPT;            // threads per row
    extern __shared__ __align__(128) unsigned char smem[];
    float *sM = reinterpret_cast<float *>(smem + L::off_m);
    float *sS = reinterpret_cast<float *>(smem + L::off_s);

    const int c = blockIdx.x, h = blockIdx.y, strip = blockIdx.z;
    const int tid = threadIdx.x;
    const int H = a.H, dv = a.dv;
    const int col0 = strip * STRIP;
    const int first = a.first ? a.first[c] : c * a.P;
    const int last = a.first ? a.first[c + 1] : (c + 1) * a.P;

    for (int idx = tid; idx < DK * STRIP; idx += CMP_THREADS) {
        int row = idx / STRIP, col = idx % STRIP;
        sS[idx] = a.S0 ? a.S0[(((size_t)c * H + h) * DK + row) * dv + col0 + col] : 0.f;
    }
    __syncthreads();

    const int row = tid / GROUPS, cg = (tid % GROUPS) * CPT;
    for (int pseg = first; pseg < last; ++pseg) {
        const size_t mh = (size_t)pseg * H + h;
        if (a.S_in) {
            for (int idx = tid; idx < DK * STRIP; idx += CMP_THREADS) {
                int rr = idx / STRIP, cc = idx % STRIP;
                a.S_in[(mh * DK + rr) * dv + col0 + cc] = sS[idx];
            }
        }
        const float *Mp = a.M + mh * DK * DK;
        for (int idx = tid; idx < DK * DK / 4; idx += CMP_THREADS) {
            int rr = idx / (DK / 4), c4 = idx % (DK / 4);
            cp_async16(&sM[rr * LDM + c4 * 4], Mp + (size_t)rr * DK + c4 * 4, true);
        }
        cp_async_commit();
        float acc[CPT];
        const float *Np = a.Nm + (mh * DK + row) * dv + col0 + cg;
#pragma unroll
        for (int u = 0; u < CPT; ++u) acc[u] = Np[u];
        cp_async_wait_all();
        __syncthreads();
#pragma unroll 4
        for (int r = 0; r < DK; ++r) {
            float m = sM[row * LDM + r];
#pragma unroll
            for (int u = 0; u < CPT; ++u) acc[u] = fmaf(m, sS[r * STRIP + cg + u], acc[u]);
        }
        __syncthreads();
#pragma unroll
        for (int u = 0; u < CPT; ++u) sS[row * STRIP + cg + u] = acc[u];
        __syncthreads();
    }
    if (a.S_final) {
        for (int idx = tid; idx < DK * STRIP; idx += CMP_THREADS) {
            int rr = idx / STRIP, cc = idx % STRIP;
            a.S_final[(((size_t)c * H + h) * DK + rr) * dv + col0 + cc] = sS[idx];
        }
    }
}

template <int DK>
static cudaError_t launch_compose_t(const ComposeArgs &a, cudaStream_t st) {
    using L = ComposeSmem<DK>;
    auto kern = kda_compose_kernel<DK>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::bytes);
    if (e != cudaSuccess) return e;
    dim3 grid(a.chains, a.H, a.dv / STRIP);
    kern<<<grid, CMP_THREADS, L::bytes, st>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_compose(const ComposeArgs &a, cudaStream_t st) {
    if (a.chains <= 0) return cudaSuccess;
    if (a.dk == 128) return launch_compose_t<128>(a, st);
    if (a.dk == 64) return launch_compose_t<64>(a, st);
    return cudaErrorInvalidValue;
}

}  // namespace kda
