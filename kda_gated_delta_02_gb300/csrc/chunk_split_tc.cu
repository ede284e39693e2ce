// chunk_split_tc.cu -- the sm_103a tensor-core prefill (dk = dv = 128, bf16
// inputs) as two kernels: the chunk-local products of every chunk at once,
// then the state walk.
//
// In the WY form of a 64-token chunk ("Noyaux KDA et FlashKDA", section
// "FlashKDA : le noyau par blocs") most of the work depends only on the
// chunk's own k, q, g and beta: the decays, the causal tiles A and B, the
// dependency inverse T = (I + A)^{-1} (fp32, "Dentro de los esfuerzos de
// optimizacion de Kimi K3", "Nota tecnica: Precision del KDA"), and the
// products W = T diag(b) K e^gamma, Q~ = Q e^gamma, K~ = K e^{gamma_63 - gamma}.
// Only U = T diag(b) V - W S, O = Q~ S + B U and S <- Diag(e^{gamma_63}) S +
// K~^T U involve the running state.  kda_chunk_prep_kernel computes the first
// group for every (chunk, head) in parallel on all SMs and leaves one operand
// blob per (chunk, head) in global memory, each tile already in the swizzled
// shared-memory layout of its tensor-core operand; kda_chunk_walk_kernel walks
// each (segment, head) unit with one bulk copy of the blob per chunk and only
// the state-dependent products on its critical path.  Both kernels use the same
// arithmetic as the single-kernel version (chunk_fwd_tc.cu), operation for
// operation, so the two paths give identical results.
//
// Chunk slots: the chunks of unit u (token range [t0, t1)) occupy slots
// floor(t0 / 64) + u + j, j < ceil((t1 - t0) / 64).  Units come in token order
// with disjoint ranges, so these slot ranges are disjoint and all lie below
// floor(T / 64) + units.  The blob area holds a window of slots (a "piece");
// a unit that crosses a piece boundary hands its state to the next piece
// through a carry buffer (at most one unit crosses each boundary).
//
// The backward (chunk_bwd_tc.cu) runs these kernels as its forward pass:
// kda_chunk_prep_aux_kernel also keeps every (chunk, head)'s fp32 T and M^T,
// and the walk can save its bf16 S^T and U^T operand tiles of every chunk by
// bulk copies (with or without the outputs).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_umma.cuh"

namespace kda {
namespace sp {

constexpr int D = 128;
constexpr int CH = 64;
constexpr uint32_t WAIT_LIMIT = 1u << 24;
// The bound of the walk's first wait (on its first chunk's copy).  A test
// build (KDA_TEST_SHORT_FIRST_WAIT) gives up on it at once, to exercise the
// timeout path: status reported, the copy still in flight drained (full
// bound), memory released.  The library itself uses the full bound.
#ifdef KDA_TEST_SHORT_FIRST_WAIT
constexpr uint32_t FIRST_WAIT_LIMIT = 0;
#else
constexpr uint32_t FIRST_WAIT_LIMIT = WAIT_LIMIT;
#endif

// operand blob of one (chunk, head): byte offsets, every tile 1024-aligned
constexpr uint32_t BL_W = kBlobW;      // W, MN-major (128 key rows i x 64 tokens t)     bf16
constexpr uint32_t BL_TB = kBlobTB;    // T diag(b), K-major 64 x 64                     bf16
constexpr uint32_t BL_QT = kBlobQT;    // Q e^gamma, K-major 64 x 128                     bf16
constexpr uint32_t BL_KT = kBlobKT;    // K e^{gamma_63 - gamma}, MN-major (s x dk)        bf16
constexpr uint32_t BL_BM = kBlobBM;    // B, K-major 64 x 64 (masked, diagonal included)  bf16
constexpr uint32_t BL_GAM = kBlobGam;  // e^{gamma_63} per key channel                     f32 [128]
static_assert(BL_GAM + 512 == kChunkBlobBytes, "blob layout");

// rows of R_i start at row 8 i (i+1): 0, 16, 48, 96 (16 (i+1) rows each)
__host__ __device__ constexpr uint32_t r_row(int i) { return 8u * (uint32_t)(i * (i + 1)); }

// ============================================================================ unit ranges
// Token range of work unit `unit` (a sequence in SEQ mode, a segment
// otherwise); false when the unit does not exist or its range is invalid.
__device__ __forceinline__ bool unit_range(const ChunkArgs &p, int unit, int &n, int &t0, int &t1, bool &last) {
    last = true;
    if (p.mode == MODE_SEQ) {
        n = unit;
        t0 = p.cu_seqlens[n];
        t1 = p.cu_seqlens[n + 1];
        return !(t0 < 0 || t1 < t0 || t1 > p.T);
    }
    if (p.seg_table) {
        if (unit >= *p.seg_count) return false;
        const int4 e = reinterpret_cast<const int4 *>(p.seg_table)[unit];
        n = e.x;
        t0 = e.y;
        t1 = e.z;
        last = e.w != 0;
        return true;
    }
    n = 0;
    t0 = unit * p.seg_len;
    t1 = min(p.T, t0 + p.seg_len);
    last = t1 == p.T;
    return true;
}

// slot list: slot -> {first token, length}; slots of no chunk keep length 0
__global__ void kda_chunk_list_kernel(const ChunkArgs p, int nslots, int2 *list) {
    int n, t0, t1;
    bool last;
    const int unit = blockIdx.x;
    if (!unit_range(p, unit, n, t0, t1, last)) return;
    const int base = t0 / CH + unit, nch = (t1 - t0 + CH - 1) / CH;
    for (int j = threadIdx.x; j < nch; j += blockDim.x) {
        const int s = base + j;
        if (s < nslots) list[s] = make_int2(t0 + CH * j, min(CH, t1 - t0 - CH * j));
    }
}

// ============================================================================ chunk-local pass
constexpr int NT1 = 256;
// shared memory (bytes from a 1024-aligned base); two CTAs per SM
constexpr uint32_t P_L = 0;          // L = [k x ; q x] of each 16-token block, K-major 128 rows x 128
constexpr uint32_t P_R = 32768;      // R = [R_0; R_1; R_2; R_3], K-major 160 rows x 128
constexpr uint32_t R_KB = 160 * 128; //   its K-block stride
constexpr uint32_t P_AF = 0;         // A fp32 [64][68] (over L, R once their product is done)
constexpr uint32_t P_TF = 17408;     // T fp32 [64][68]
constexpr uint32_t P_KG = 73728;     // K e^gamma, MN-major (s x dk)
constexpr uint32_t P_TB = 90112;     // T diag(b), K-major 64 x 64
constexpr uint32_t P_BETA = 98304;   // f32 [64]
constexpr uint32_t P_PART = 98560;   // f32 [2][4][128] half-block products
constexpr uint32_t P_BAR = 102656;   // 2 mbarriers: A/B product, W product
constexpr uint32_t P_TMEM = 102672;  // tensor-memory base address
constexpr uint32_t P_CLAIM = 102676; // items claimed by thread 0 (2 ints)
constexpr uint32_t P_SMEM = 102688 + 1024;
constexpr int LDF = 68;
constexpr uint32_t TM1_AB = 0, TM1_W = 160;  // 224 of 256 columns

struct PrepParams {
    const void *q, *k;   // bf16 [T][H][128]
    const float *g;      // f32 [T][H][128]
    const float *beta;   // f32 [T][H]
    int H;
    float g_min;
    CUtensorMap tq, tk, tg, tb;  // q, k, g boxes of 64 tokens x 1 head x 128; beta box of 64 tokens x 4 heads
    const int2 *list;    // slot -> {first token, length}
    int slot0;           // first slot of this launch
    int nitems;          // (slot1 - slot0) * H items, w = (slot - slot0) * H + h
    int *claim;          // item counter of this launch, zero at launch; CTAs claim items in order
    unsigned char *blob; // [w][kChunkBlobBytes]
    float *aux;          // backward's forward pass only: [w][2][64][64] T (row t) and M^T (row s)
    int need_q;          // 0: transitions only (no Q~, no B)
    int pf_beta;         // tb is encoded (H a multiple of 4)
    uint32_t *status;
};

// The body of the chunk-local kernel.  AUX (the forward pass that a backward
// runs) also keeps, per item, the fp32 dependency inverse T and the strictly
// lower tile M = (K x)(K / x)^T before the beta scaling, which the backward's
// chunk kernel needs and the blob does not hold.
template <bool AUX>
__device__ __forceinline__ void prep_body(const PrepParams &p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(sm);
    const uint32_t sb4 = sb >> 4;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = p.H, nitems = p.nitems;
    float *sBeta = reinterpret_cast<float *>(sm + P_BETA);
    float *sPart = reinterpret_cast<float *>(sm + P_PART);
    const uint32_t bar_ab = sb + P_BAR, bar_w = sb + P_BAR + 8;
    const bool need_q = p.need_q != 0;
    const float g_min = p.g_min;

    if (tid == 0) {
        umma::mbar_init(bar_ab, 1);
        umma::mbar_init(bar_w, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == 0) umma::tmem_alloc(sb + P_TMEM, 256);
    umma::fence_before();
    __syncthreads();
    umma::fence_after();
    const uint32_t tmem = *reinterpret_cast<const uint32_t *>(sm + P_TMEM);
    const int qd = warp & 3;  // TMEM lane quadrant of this warp
    const uint32_t tq = tmem + ((uint32_t)(32 * qd) << 16);

    // Items w = (slot - slot0) * H + h, claimed in increasing order from the
    // launch's counter, so CTAs that start late (the SMs were busy with other
    // work) take fewer items and the blobs are written roughly in slot order.
    // Each CTA holds the item it works on and the next one it claimed: while
    // item w runs, the rows of the next item are prefetched into L2 (its chunk
    // entry was read one item earlier), so its loads do not wait on DRAM.
    int *sClaim = reinterpret_cast<int *>(sm + P_CLAIM);
    bool alive = true;
    uint32_t it = 0;  // items processed (mbarrier parity)
    if (tid == 0) {
        const int w0 = atomicAdd(p.claim, 1);
        sClaim[0] = w0;
        sClaim[1] = atomicAdd(p.claim, 1);
    }
    __syncthreads();
    int w = sClaim[0], wn = sClaim[1];
    int2 cl = (w < nitems) ? p.list[p.slot0 + w / H] : make_int2(0, 0);
    int2 ncl = (wn < nitems) ? p.list[p.slot0 + wn / H] : make_int2(0, 0);
    __syncthreads();  // claims read before thread 0 writes the next one

    while (w < nitems) {
    const int h = w % H;
    const int tc = cl.x, Lc = cl.y;
    int wnn;
    {
        if (tid == 0) {
            sClaim[0] = (wn < nitems) ? atomicAdd(p.claim, 1) : nitems;
            if (wn < nitems && ncl.y > 0) {
                const int hn = wn % H;
                if (need_q) umma::prefetch_tile_3d(&p.tq, 0, hn, ncl.x);
                umma::prefetch_tile_3d(&p.tk, 0, hn, ncl.x);
                umma::prefetch_tile_3d(&p.tg, 0, hn, ncl.x);
                if (p.pf_beta) umma::prefetch_tile_2d(&p.tb, hn & ~3, ncl.x);
            }
        }
        __syncthreads();
        wnn = sClaim[0];
    }
    const int2 nncl = (wnn < nitems) ? p.list[p.slot0 + wnn / H] : make_int2(0, 0);
    if (Lc > 0) {
    unsigned char *out = p.blob + ((size_t)w * kChunkBlobBytes);

    // ---------------------------------------------------------------- loads
    // warp w = half block (block i = w / 2, half hf = w % 2, tokens 8 w .. 8 w + 7),
    // lane = channel quad (channels 4 lane .. 4 lane + 3); rows past the chunk
    // end read as zero (g = 0 -> e = 1)
    const int i = warp >> 1, hf = warp & 1, ch = 4 * lane, tb = 8 * warp;
    float4 e[8];
    uint2 kraw[8], qraw[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        const int t = tb + r;
        const bool ok = t < Lc;
        const size_t row = ((size_t)(tc + t) * H + h) * D;  // element offset of the token's row
        e[r] = ok ? __ldg(reinterpret_cast<const float4 *>(p.g + row) + lane) : make_float4(0.f, 0.f, 0.f, 0.f);
        kraw[r] = ok ? __ldg(reinterpret_cast<const uint2 *>(reinterpret_cast<const __nv_bfloat16 *>(p.k) + row) + lane)
                     : make_uint2(0u, 0u);
        qraw[r] = (ok && need_q)
                      ? __ldg(reinterpret_cast<const uint2 *>(reinterpret_cast<const __nv_bfloat16 *>(p.q) + row) + lane)
                      : make_uint2(0u, 0u);
    }
    if (tid < CH) sBeta[tid] = (tid < Lc) ? p.beta[(size_t)(tc + tid) * H + h] : 0.f;

    // ---------------------------------------------------------------- decays
    // running products of e^{g} inside each 8-token half block, combined as in
    // the single-kernel version: x_t = prod_{block start <= r <= t}, y_t =
    // prod_{t < r <= block end}, delta_i = block product
#pragma unroll
    for (int r = 0; r < 8; ++r) {
        e[r].x = __expf(fmaxf(e[r].x, g_min));
        e[r].y = __expf(fmaxf(e[r].y, g_min));
        e[r].z = __expf(fmaxf(e[r].z, g_min));
        e[r].w = __expf(fmaxf(e[r].w, g_min));
    }
    // four products as two packed f32x2 multiplies (each lane rounds like a scalar multiply)
    auto mul4 = [](float4 a, float4 b) {
        const float2 lo = __fmul2_rn(make_float2(a.x, a.y), make_float2(b.x, b.y));
        const float2 hi = __fmul2_rn(make_float2(a.z, a.w), make_float2(b.z, b.w));
        return make_float4(lo.x, lo.y, hi.x, hi.y);
    };
    {
        float4 ph = make_float4(1.f, 1.f, 1.f, 1.f);
#pragma unroll
        for (int r = 0; r < 8; ++r) {  // (scalar: packed here costs registers)
            ph.x *= e[r].x;
            ph.y *= e[r].y;
            ph.z *= e[r].z;
            ph.w *= e[r].w;
        }
        *reinterpret_cast<float4 *>(sPart + (hf * 4 + i) * 128 + ch) = ph;
    }
    __syncthreads();
    float4 dl[4], pz;  // block decays; the other half's product for this thread's half
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        const float4 a0 = *reinterpret_cast<const float4 *>(sPart + (0 * 4 + m) * 128 + ch);
        const float4 a1 = *reinterpret_cast<const float4 *>(sPart + (1 * 4 + m) * 128 + ch);
        dl[m] = mul4(a0, a1);
        if (m == i) pz = hf ? a0 : a1;
    }
    float4 gb = make_float4(1.f, 1.f, 1.f, 1.f), cc = gb;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        if (m < i) gb = mul4(gb, dl[m]);
        if (m > i) cc = mul4(cc, dl[m]);
    }
    if (warp == 0)
        *reinterpret_cast<float4 *>(out + BL_GAM + ch * 4) = mul4(mul4(mul4(dl[0], dl[1]), dl[2]), dl[3]);
    // right-operand factors for row blocks i2 >= i: 1/delta_i (i2 == i), c_{i2,i} otherwise
    float4 vf[4];
#pragma unroll
    for (int i2 = 0; i2 < 4; ++i2) {
        float4 f = make_float4(1.f, 1.f, 1.f, 1.f);
        if (i2 == i) {
            f = make_float4(__frcp_rn(dl[i].x), __frcp_rn(dl[i].y), __frcp_rn(dl[i].z), __frcp_rn(dl[i].w));
        } else {
#pragma unroll
            for (int m = 0; m < 4; ++m)
                if (m > i && m < i2) f = mul4(f, dl[m]);
        }
        vf[i2] = f;
    }

    // ---------------------------------------------------------------- operands
    // Every destination row of token r has (row & 7) == r: one swizzled column
    // offset per r serves all operands; each lane stores 8 bytes (4 channels).
    // L, R and K e^gamma stay in shared memory (operands here); Q~ and K~ go
    // straight to the blob.  x-side operands in a forward pass, y-side ones in
    // a backward pass (x_t and y_t are running products in opposite directions).
    {
        const uint32_t c8 = (uint32_t)(ch & 63) >> 3, lo = (uint32_t)(ch & 7) << 1, kb = (uint32_t)ch >> 6;
        const uint32_t aL = sb + P_L + kb * 16384u + (uint32_t)(32 * i + 8 * hf) * 128u;
        const uint32_t aRk = sb + P_R + kb * R_KB + (uint32_t)tb * 128u;
        const uint32_t atom = ((uint32_t)warp * 2u + kb) * 1024u;
        const uint32_t aKG = sb + P_KG + atom;
        unsigned char *gKT = out + BL_KT + atom;
        unsigned char *gQT = out + BL_QT + kb * 8192u + (uint32_t)tb * 128u;
        auto pk2 = [](float4 v) { return make_uint2(pack_bf16(v.x, v.y), pack_bf16(v.z, v.w)); };
        float4 pr = make_float4(1.f, 1.f, 1.f, 1.f);
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const uint32_t o = (uint32_t)r * 128u + ((c8 ^ (uint32_t)r) << 4) + lo;
            pr = mul4(pr, e[r]);
            const float4 x = hf ? mul4(pr, pz) : pr;
            const float2 k01 = unpack_bf16(kraw[r].x), k23 = unpack_bf16(kraw[r].y);
            const float4 lk = mul4(make_float4(k01.x, k01.y, k23.x, k23.y), x);
            const uint2 lkp = pk2(lk), kgp = pk2(mul4(lk, gb));
            sts64(aL + o, lkp.x, lkp.y);
            sts64(aKG + o, kgp.x, kgp.y);
            const float2 q01 = unpack_bf16(qraw[r].x), q23 = unpack_bf16(qraw[r].y);
            const float4 lq = mul4(make_float4(q01.x, q01.y, q23.x, q23.y), x);
            const uint2 lqp = pk2(lq);
            sts64(aL + 2048u + o, lqp.x, lqp.y);
            if (need_q) *reinterpret_cast<uint2 *>(gQT + o) = pk2(mul4(lq, gb));
        }
        float4 sf = make_float4(1.f, 1.f, 1.f, 1.f);
#pragma unroll
        for (int r = 7; r >= 0; --r) {
            const uint32_t o = (uint32_t)r * 128u + ((c8 ^ (uint32_t)r) << 4) + lo;
            const float4 y = hf ? sf : mul4(sf, pz);
            const float2 k01 = unpack_bf16(kraw[r].x), k23 = unpack_bf16(kraw[r].y);
            const float4 ky = mul4(make_float4(k01.x, k01.y, k23.x, k23.y), y);
            uint2 v;
            if (i <= 0) { v = pk2(mul4(ky, vf[0])); sts64(aRk + r_row(0) * 128u + o, v.x, v.y); }
            if (i <= 1) { v = pk2(mul4(ky, vf[1])); sts64(aRk + r_row(1) * 128u + o, v.x, v.y); }
            if (i <= 2) { v = pk2(mul4(ky, vf[2])); sts64(aRk + r_row(2) * 128u + o, v.x, v.y); }
            v = pk2(mul4(ky, vf[3]));
            sts64(aRk + r_row(3) * 128u + o, v.x, v.y);
            *reinterpret_cast<uint2 *>(gKT + o) = pk2(mul4(ky, cc));
            sf = mul4(sf, e[r]);
        }
    }
    umma::fence_proxy_async();
    __syncthreads();

    // ---------------------------------------------------------------- A and B tiles
    // one M = 128, N = 160 product: block i reads its 32 L rows (TMEM lane
    // quadrant i) against its R_i columns
    if (tid == 0) {
        umma::fence_after();
        constexpr uint32_t id = umma::idesc_bf16(128, 160, 0, 0, 0);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint32_t kb = ks >> 2, kin = (ks & 3) * 32;
            const uint64_t a = umma::sdesc4(sb4 + ((P_L + kb * 16384 + kin) >> 4), 16, 1024);
            const uint64_t b = umma::sdesc4(sb4 + ((P_R + kb * R_KB + kin) >> 4), 16, 1024);
            umma::mma(tmem + TM1_AB, a, b, id, ks > 0 ? 1u : 0u);
        }
        umma::commit(bar_ab);
    }
    bool ok = umma::mbar_wait(bar_ab, it & 1u, WAIT_LIMIT);
    ok = __syncthreads_and(ok) != 0;
    const bool w_issued = ok;  // the W product is issued exactly when the A/B product landed
    const uint32_t par = it & 1u;
    umma::fence_after();

    if (ok) {
        // A (fp32, scaled by b_t, strictly lower) into shared memory; B (bf16,
        // diagonal included) into the blob.  Lane quadrant i = block i: lanes
        // 0-15 the key rows t = 16 i + l, 16-31 the query rows; column groups
        // cg = warp / 4 and cg + 2 of R_i (zero where cg > i).
        float *sAf = reinterpret_cast<float *>(sm + P_AF);
        const int t = 16 * qd + (lane & 15);
        const bool is_q = lane >= 16;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int cg = (warp >> 2) + 2 * u, s0 = 16 * cg;
            float v[16];
            if (cg <= qd) {
                umma::ld16(tq + TM1_AB + r_row(qd) + 16 * cg, v);
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = 0.f;
            }
            if (!is_q) {
                if constexpr (AUX) {  // M^T [s][t], strictly lower M, zero elsewhere
                    float *mt = p.aux + (size_t)w * 8192 + 4096;
#pragma unroll
                    for (int j = 0; j < 16; ++j) mt[(s0 + j) * 64 + t] = (s0 + j < t) ? v[j] : 0.f;
                }
                if (cg <= qd) {
                    const float2 bt2 = make_float2(sBeta[t], sBeta[t]);
#pragma unroll
                    for (int j = 0; j < 16; j += 4) {
                        const float2 a01 = __fmul2_rn(bt2, make_float2(v[j], v[j + 1]));
                        const float2 a23 = __fmul2_rn(bt2, make_float2(v[j + 2], v[j + 3]));
                        *reinterpret_cast<float4 *>(sAf + t * LDF + s0 + j) =
                            make_float4((s0 + j < t) ? a01.x : 0.f, (s0 + j + 1 < t) ? a01.y : 0.f,
                                        (s0 + j + 2 < t) ? a23.x : 0.f, (s0 + j + 3 < t) ? a23.y : 0.f);
                    }
                }
            } else if (need_q) {
                uint32_t bp[8];
#pragma unroll
                for (int j = 0; j < 16; j += 2)
                    bp[j >> 1] = pack_bf16((s0 + j <= t) ? v[j] : 0.f, (s0 + j + 1 <= t) ? v[j + 1] : 0.f);
                unsigned char *row = out + BL_BM + (uint32_t)t * 128u;
                const uint32_t sw = (uint32_t)(t & 7);
                *reinterpret_cast<uint4 *>(row + (((2u * cg) ^ sw) << 4)) = make_uint4(bp[0], bp[1], bp[2], bp[3]);
                *reinterpret_cast<uint4 *>(row + (((2u * cg + 1u) ^ sw) << 4)) = make_uint4(bp[4], bp[5], bp[6], bp[7]);
            }
        }
    }
    __syncthreads();

    // ---------------------------------------------------------------- T = (I + A)^{-1}, fp32
    if (ok) {
        float *sAf = reinterpret_cast<float *>(sm + P_AF);
        float *sTf = reinterpret_cast<float *>(sm + P_TF);
        // diagonal 16 x 16 blocks by substitution with one column per lane in
        // registers (lanes 0-15 of warp 2 + w -> block 2w, 16-31 -> 2w+1), row by
        // row: T[r][c] = delta_rc - sum_{m < r} A[r][m] T[m][c], the terms added in
        // increasing m; the rows of A come in 16-byte loads
        if (warp == 2 || warp == 3) {
            const int bi = 2 * (warp - 2) + (lane >> 4), c = lane & 15;
            const float *Ab = sAf + (16 * bi) * LDF + 16 * bi;
            float acc[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float v = (r == c) ? 1.f : 0.f;
#pragma unroll
                for (int m4 = 0; m4 < r; m4 += 4) {
                    const float4 a4 = *reinterpret_cast<const float4 *>(Ab + r * LDF + m4);
                    v = fmaf(-a4.x, acc[m4], v);
                    if (m4 + 1 < r) v = fmaf(-a4.y, acc[m4 + 1], v);
                    if (m4 + 2 < r) v = fmaf(-a4.z, acc[m4 + 2], v);
                    if (m4 + 3 < r) v = fmaf(-a4.w, acc[m4 + 3], v);
                }
                acc[r] = v;
            }
            float *Tb = sTf + (16 * bi) * LDF + 16 * bi;
#pragma unroll
            for (int r = 0; r < 16; ++r) Tb[r * LDF + c] = acc[r];
        }
        __syncthreads();
        // 32 x 32 diagonal halves: T_10 = -T_11 A_10 T_00, T_32 = -T_33 A_32 T_22;
        // X = A_10 T_00 goes to the (unused) upper block (0,1) of the A scratch.
        // Thread (half hb, row r, column quad cq) of the first 128 forms four
        // outputs from 16-byte loads (even and odd m summed apart, then added).
        {
            const int hb = (tid >> 6) & 1, r = (tid >> 2) & 15, c0 = 4 * (tid & 3);
            const int bi = 2 * hb + 1, bj = 2 * hb;
            // packed f32x2 fused multiply-adds and adds (each lane rounds like the scalar op)
            auto fma4 = [](float a, float4 b, float4 acc) {
                const float2 a2 = make_float2(a, a);
                const float2 lo = __ffma2_rn(a2, make_float2(b.x, b.y), make_float2(acc.x, acc.y));
                const float2 hi = __ffma2_rn(a2, make_float2(b.z, b.w), make_float2(acc.z, acc.w));
                return make_float4(lo.x, lo.y, hi.x, hi.y);
            };
            auto add4 = [](float4 a, float4 b) {
                const float2 lo = __fadd2_rn(make_float2(a.x, a.y), make_float2(b.x, b.y));
                const float2 hi = __fadd2_rn(make_float2(a.z, a.w), make_float2(b.z, b.w));
                return make_float4(lo.x, lo.y, hi.x, hi.y);
            };
            if (tid < 128) {
                const float *Ar = sAf + (16 * bi + r) * LDF + 16 * bj;
                const float *Tc = sTf + (16 * bj) * LDF + 16 * bj + c0;
                float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
#pragma unroll
                for (int m4 = 0; m4 < 16; m4 += 4) {
                    const float4 a4 = *reinterpret_cast<const float4 *>(Ar + m4);
                    x0 = fma4(a4.x, *reinterpret_cast<const float4 *>(Tc + (m4 + 0) * LDF), x0);
                    x1 = fma4(a4.y, *reinterpret_cast<const float4 *>(Tc + (m4 + 1) * LDF), x1);
                    x0 = fma4(a4.z, *reinterpret_cast<const float4 *>(Tc + (m4 + 2) * LDF), x0);
                    x1 = fma4(a4.w, *reinterpret_cast<const float4 *>(Tc + (m4 + 3) * LDF), x1);
                }
                *reinterpret_cast<float4 *>(sAf + (16 * bj + r) * LDF + 16 * bi + c0) = add4(x0, x1);
                *reinterpret_cast<float4 *>(sTf + (16 * bj + r) * LDF + 16 * bi + c0) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            __syncthreads();
            if (tid < 128) {
                const float *Ti = sTf + (16 * bi + r) * LDF + 16 * bi;
                const float *Xs = sAf + (16 * bj) * LDF + 16 * bi + c0;
                float4 y0 = make_float4(0.f, 0.f, 0.f, 0.f), y1 = y0;
#pragma unroll
                for (int m4 = 0; m4 < 16; m4 += 4) {
                    const float4 t4 = *reinterpret_cast<const float4 *>(Ti + m4);
                    y0 = fma4(t4.x, *reinterpret_cast<const float4 *>(Xs + (m4 + 0) * LDF), y0);
                    y1 = fma4(t4.y, *reinterpret_cast<const float4 *>(Xs + (m4 + 1) * LDF), y1);
                    y0 = fma4(t4.z, *reinterpret_cast<const float4 *>(Xs + (m4 + 2) * LDF), y0);
                    y1 = fma4(t4.w, *reinterpret_cast<const float4 *>(Xs + (m4 + 3) * LDF), y1);
                }
                const float4 y = add4(y0, y1);
                *reinterpret_cast<float4 *>(sTf + (16 * bi + r) * LDF + 16 * bj + c0) = make_float4(-y.x, -y.y, -y.z, -y.w);
            }
            __syncthreads();
        }
        // lower-left 32 x 32: T_21 = -T_22 (A_21 T_11), two 32x32x32 fp32
        // products as tf32 tensor products with hi/lo splits (3 MMAs per step);
        // warp w owns the 16 x 8 tile (rows 16 (w >> 2), cols 8 (w & 3)); the
        // intermediate X goes to the unused upper-right 32 x 32 of the A scratch
        // and the result straight into T diag(b) as bf16
        {
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
            float *X64 = sAf + 32;  // rows 0-31, columns 32-63
            product(sAf + 32 * LDF, sTf, acc);  // X = A_21 T_11
            float *Xt = X64 + (16 * mt + gq) * LDF + 8 * nt + 2 * q4;
            *reinterpret_cast<float2 *>(Xt) = make_float2(acc[0], acc[1]);
            *reinterpret_cast<float2 *>(Xt + 8 * LDF) = make_float2(acc[2], acc[3]);
            __syncthreads();
            product(sTf + 32 * LDF + 32, X64, acc);  // T_22 X
            const int t = 32 + 16 * mt + gq, s0 = 8 * nt + 2 * q4;
            if constexpr (AUX) {  // T_21 = -T_22 X in fp32
                float *ta = p.aux + (size_t)w * 8192;
                *reinterpret_cast<float2 *>(ta + t * 64 + s0) = make_float2(-acc[0], -acc[1]);
                *reinterpret_cast<float2 *>(ta + (t + 8) * 64 + s0) = make_float2(-acc[2], -acc[3]);
            }
            const float b0 = sBeta[s0], b1 = sBeta[s0 + 1];
            *reinterpret_cast<uint32_t *>(sm + P_TB + umma::kmaj(t, s0, 64)) = pack_bf16(-acc[0] * b0, -acc[1] * b1);
            *reinterpret_cast<uint32_t *>(sm + P_TB + umma::kmaj(t + 8, s0, 64)) = pack_bf16(-acc[2] * b0, -acc[3] * b1);
        }
        // T diag(b) for the rest, 8 columns per step: rows 0-31 (all 64 columns),
        // rows 32-63 columns 32-63; zero above the diagonal
        for (int e2 = tid; e2 < 384; e2 += NT1) {
            int t, s0;
            if (e2 < 256) {
                t = e2 >> 3;
                s0 = 8 * (e2 & 7);
            } else {
                t = 32 + ((e2 - 256) >> 2);
                s0 = 32 + 8 * ((e2 - 256) & 3);
            }
            const float4 ta = *reinterpret_cast<const float4 *>(sTf + t * LDF + s0);
            const float4 tb4 = *reinterpret_cast<const float4 *>(sTf + t * LDF + s0 + 4);
            const float4 ba = *reinterpret_cast<const float4 *>(sBeta + s0);
            const float4 bb = *reinterpret_cast<const float4 *>(sBeta + s0 + 4);
            const float2 v01 = __fmul2_rn(make_float2(ta.x, ta.y), make_float2(ba.x, ba.y));
            const float2 v23 = __fmul2_rn(make_float2(ta.z, ta.w), make_float2(ba.z, ba.w));
            const float2 v45 = __fmul2_rn(make_float2(tb4.x, tb4.y), make_float2(bb.x, bb.y));
            const float2 v67 = __fmul2_rn(make_float2(tb4.z, tb4.w), make_float2(bb.z, bb.w));
            const float v[8] = {v01.x, v01.y, v23.x, v23.y, v45.x, v45.y, v67.x, v67.y};
            uint32_t pk[4];
#pragma unroll
            for (int j = 0; j < 8; j += 2)
                pk[j >> 1] = pack_bf16((s0 + j <= t) ? v[j] : 0.f, (s0 + j + 1 <= t) ? v[j + 1] : 0.f);
            *reinterpret_cast<uint4 *>(sm + P_TB + umma::kmaj(t, s0, 64)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            if constexpr (AUX) {  // the same blocks of T in fp32, zero above the diagonal
                float *dst = p.aux + (size_t)w * 8192 + t * 64 + s0;
                *reinterpret_cast<float4 *>(dst) = make_float4((s0 <= t) ? ta.x : 0.f, (s0 + 1 <= t) ? ta.y : 0.f,
                                                              (s0 + 2 <= t) ? ta.z : 0.f, (s0 + 3 <= t) ? ta.w : 0.f);
                *reinterpret_cast<float4 *>(dst + 4) =
                    make_float4((s0 + 4 <= t) ? tb4.x : 0.f, (s0 + 5 <= t) ? tb4.y : 0.f, (s0 + 6 <= t) ? tb4.z : 0.f,
                                (s0 + 7 <= t) ? tb4.w : 0.f);
            }
        }
    }
    umma::fence_proxy_async();
    __syncthreads();

    // ---------------------------------------------------------------- W^T = (K e^gamma)^T (T diag b)^T
    if (ok && tid == 0) {
        umma::fence_after();
        constexpr uint32_t id = umma::idesc_bf16(128, 64, 1, 0, 0);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            const uint64_t b = umma::sdesc4(sb4 + ((P_TB + ks * 32) >> 4), 16, 1024);
            umma::mma(tmem + TM1_W, umma::sdesc4(sb4 + ((P_KG + ks * 4096) >> 4), 1024, 2048), b, id, ks > 0 ? 1u : 0u);
        }
        umma::commit(bar_w);
    }
    if (ok) {
        // T diag(b) into the blob while the product runs (both only read it)
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int idx = tid + u * NT1;
            *reinterpret_cast<uint4 *>(out + BL_TB + idx * 16) = *reinterpret_cast<const uint4 *>(sm + P_TB + idx * 16);
        }
        ok = umma::mbar_wait(bar_w, it & 1u, WAIT_LIMIT);
    }
    ok = __syncthreads_and(ok) != 0;
    umma::fence_after();
    if (ok) {
        // W as an MN-major operand (n = t, k = key channel i = TMEM lane)
        const int ich = 32 * qd + lane;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int cg = 2 * (warp >> 2) + u;
            float v[16];
            umma::ld16(tq + TM1_W + 16 * cg, v);
            *reinterpret_cast<uint4 *>(out + BL_W + umma::mnmaj(16 * cg, ich, 1)) =
                make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
            *reinterpret_cast<uint4 *>(out + BL_W + umma::mnmaj(16 * cg + 8, ich, 1)) =
                make_uint4(pack_bf16(v[8], v[9]), pack_bf16(v[10], v[11]), pack_bf16(v[12], v[13]),
                           pack_bf16(v[14], v[15]));
        }
    }
    umma::fence_before();
    __syncthreads();
    ++it;
    if (!ok) {  // uniform: leave once the products still in flight are done with tensor memory
        umma::mbar_wait(bar_ab, par, WAIT_LIMIT);
        if (w_issued) umma::mbar_wait(bar_w, par, WAIT_LIMIT);
        alive = false;
        break;
    }
    }  // Lc > 0
    __syncthreads();  // the claim was read by every thread before thread 0 writes the next
    w = wn;
    wn = wnn;
    cl = ncl;
    ncl = nncl;
    }  // items
    if (!alive && tid == 0) report_status(p.status, KDA_STATUS_TIMEOUT);
    if (warp == 0) umma::tmem_dealloc(tmem, 256);
    // launched as a programmatic dependent of a walk: finish only after that
    // walk has, so the next walk on the stream (which waits for this launch)
    // also follows it (a no-op for an ordinary launch)
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

__global__ void __launch_bounds__(NT1, 2) kda_chunk_prep_kernel(const __grid_constant__ PrepParams p) {
    prep_body<false>(p);
}
__global__ void __launch_bounds__(NT1, 2) kda_chunk_prep_aux_kernel(const __grid_constant__ PrepParams p) {
    prep_body<true>(p);
}

// ============================================================================ state walk
constexpr int NT2 = 512;
constexpr uint32_t W_BUF = 0;           // two operand blobs (double buffer)
constexpr uint32_t W_BUFSTRIDE = 66560;
constexpr uint32_t W_V = 133120;        // two V tiles (MN-major s x dv: two 64-wide halves of [64 s][128 B])
constexpr uint32_t W_ST = 165888;       // S^T bf16, K-major 128 x 128
constexpr uint32_t W_UT = 198656;       // U^T bf16, K-major 128 x 64; then the output stage [64][128] bf16
constexpr uint32_t W_BAR = 215040;      // 4 mbarriers: buffer 0, buffer 1, U product, O / state products
constexpr uint32_t W_TMEM = 215072;
constexpr uint32_t W_SMEM = 215088 + 1024;
constexpr uint32_t TM_ST = 0, TM_U = 128, TM_O = 192;  // 256 columns

struct WalkParams {
    ChunkArgs a;
    CUtensorMap tv;              // v [T][H][dv] bf16, box 64 x 1 x 64, 128-byte swizzle
    const unsigned char *blob;   // blobs of slots [slot0, slot1)
    int slot0, slot1;
    const float *carry_in;       // [tiles][H][128][128]: state of the unit cut at slot0
    float *carry_out;            // state of the unit cut at slot1
    // backward's forward pass: per (slot, head) the bf16 operand tiles the walk
    // builds, S^T at the chunk start (K-major 128 x 128, 32 KB) and U^T
    // (K-major 128 x 64, 16 KB), indexed by absolute slot; null for none
    unsigned char *save_s, *save_u;
};

__global__ void __launch_bounds__(NT2, 1) kda_chunk_walk_kernel(const __grid_constant__ WalkParams P) {
    const ChunkArgs &p = P.a;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(sm);
    const uint32_t sb4 = sb >> 4;
    const uint32_t bar0 = sb + W_BAR, bar_u = bar0 + 16, bar_o = bar0 + 24;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int unit = blockIdx.x, h = blockIdx.y, tile = blockIdx.z;
    const int H = p.H, dv = p.dv;
    // a chunk-local launch that follows on the stream as a programmatic
    // dependent may start once every CTA of this walk is resident: it reads
    // nothing this walk writes
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

    // ---------------------------------------------------------------- work unit and its chunks in this piece
    int n, t0, t1;
    bool last_seg;
    if (!unit_range(p, unit, n, t0, t1, last_seg)) {
        if (p.mode == MODE_SEQ && tid == 0 && P.slot0 == 0) report_status(p.status, KDA_STATUS_BAD_SEQLENS);
        return;
    }
    const int nch = (t1 - t0 + CH - 1) / CH, sbase = t0 / CH + unit;
    int jb, je;
    if (nch == 0) {  // an empty unit carries its state in the piece that holds its first slot
        if (sbase < P.slot0 || sbase >= P.slot1) return;
        jb = je = 0;
    } else {
        jb = max(0, P.slot0 - sbase);
        je = min(nch, P.slot1 - sbase);
        if (jb >= je) return;
    }
    const bool cut_in = jb > 0, cut_out = je < nch;
    const int seq0 = (p.mode == MODE_SEQ) ? t0 : ((p.seg_table && p.cu_seqlens) ? p.cu_seqlens[n] : 0);
    const bool transition = p.mode == MODE_TRANSITION;
    const bool m_part = transition && tile == 0;  // augmented columns [0, dk): M
    const bool has_v = !m_part;
    const bool need_q = !transition && p.o != nullptr;  // outputs wanted
    const bool save = P.save_s != nullptr;
    const int vcol0 = transition ? 0 : tile * D;

    // ---------------------------------------------------------------- setup
    if (tid == 0) {
        for (int b = 0; b < 4; ++b) umma::mbar_init(bar0 + 8 * b, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    if (warp == 0) umma::tmem_alloc(sb + W_TMEM, 256);
    umma::fence_before();
    __syncthreads();
    umma::fence_after();
    const uint32_t tmem = *reinterpret_cast<const uint32_t *>(sm + W_TMEM);

    const int qd = warp & 3, cg = warp >> 2;  // TMEM lane quadrant, column group
    const int jrow = 32 * qd + lane;          // S^T row (value column j) owned
    const uint32_t tq = tmem + ((uint32_t)(32 * qd) << 16);

    {
        float Sreg[32];
        const float *src = nullptr;
        size_t sidx = 0, ld = (size_t)dv, col0 = (size_t)vcol0;
        if (cut_in) {
            src = P.carry_in + ((size_t)tile * H + h) * D * D;
            ld = D;
            col0 = 0;
        } else if (!transition) {
            src = (p.mode == MODE_SEQ) ? p.S_init : p.S_in;
            sidx = (p.mode == MODE_SEQ) ? (size_t)n : (size_t)unit;
            if (src) src += (sidx * H + h) * D * (size_t)dv;
        }
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            const int i = 32 * cg + c;
            float v0 = 0.f;
            if (src) v0 = src[(size_t)i * ld + col0 + jrow];
            else if (m_part) v0 = (i == jrow) ? 1.f : 0.f;
            Sreg[c] = v0;
        }
        umma::st32(tq + TM_ST + 32 * cg, Sreg);
    }

    // one thread issues the copies of a chunk: the blob (one bulk copy) and V
    // (two swizzled halves; rows past the tensor end are zero-filled, rows past
    // the unit end are zeroed after arrival)
    auto issue = [&](int j, int b) {
        if (tid == 0) {
            umma::fence_proxy_async();
            const uint32_t bar = bar0 + 8 * b;
            umma::mbar_expect_tx(bar, kChunkBlobBytes + (has_v ? 16384u : 0u));
            umma::bulk_load(sb + W_BUF + b * W_BUFSTRIDE,
                            P.blob + ((size_t)(sbase + j - P.slot0) * H + h) * kChunkBlobBytes, kChunkBlobBytes, bar);
            if (has_v) {
                umma::tma_load_3d(sb + W_V + b * 16384, &P.tv, vcol0, h, t0 + CH * j, bar);
                umma::tma_load_3d(sb + W_V + b * 16384 + 8192, &P.tv, vcol0 + 64, h, t0 + CH * j, bar);
            }
        }
    };

    bool timed_out = false;
    int pend_b = -1;  // buffer with a copy in flight (the next chunk's, or one whose wait gave up)
    uint32_t pend_ph = 0;
    int pend_m = -1;  // tensor-core products whose completion wait gave up (0: U, 1: O / state)
    uint32_t pend_mph = 0;
    if (jb < je) {
        issue(jb, 0);
        pend_b = 0;
        pend_ph = 0;
    }

    for (int j = jb; j < je; ++j) {
        const int it = j - jb, b = it & 1;
        const uint32_t ph = (uint32_t)(it >> 1) & 1u, pm = (uint32_t)it & 1u;
        const int tc = t0 + CH * j, Lc = min(CH, t1 - tc);
        const uint32_t bb = W_BUF + (uint32_t)b * W_BUFSTRIDE;
        const bool landed = umma::mbar_wait(bar0 + 8 * b, ph, j == jb ? FIRST_WAIT_LIMIT : WAIT_LIMIT);
        timed_out |= !landed;
        pend_b = landed ? -1 : b;  // a copy that has not landed is still in flight
        pend_ph = ph;
        if (j + 1 < je && !timed_out) {
            issue(j + 1, b ^ 1);
            pend_b = b ^ 1;
            pend_ph = (uint32_t)((it + 1) >> 1) & 1u;
        }
        if (Lc < CH && has_v) {  // V rows (tokens) past the unit end are not ours
            for (int idx = tid; idx < (CH - Lc) * 16; idx += NT2) {
                const int r = Lc + (idx >> 4), c = idx & 15;
                *reinterpret_cast<uint4 *>(sm + W_V + b * 16384 + (c >> 3) * 8192 + umma::mnmaj(8 * (c & 7), r, 1)) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
        }
        // S^T (this thread's TMEM lane, columns 32 cg ..) as the bf16 operand of
        // the products, and the resident state decayed to the chunk end in place,
        // Diag-cols(e^{gamma_63}) S^T, onto which the U^T K~ product accumulates
        {
            const float *gam = reinterpret_cast<const float *>(sm + bb + BL_GAM);
            float Sreg[32];
            umma::ld32(tq + TM_ST + 32 * cg, Sreg);
#pragma unroll
            for (int c = 0; c < 32; c += 8) {
                uint4 pk;
                pk.x = pack_bf16(Sreg[c + 0], Sreg[c + 1]);
                pk.y = pack_bf16(Sreg[c + 2], Sreg[c + 3]);
                pk.z = pack_bf16(Sreg[c + 4], Sreg[c + 5]);
                pk.w = pack_bf16(Sreg[c + 6], Sreg[c + 7]);
                *reinterpret_cast<uint4 *>(sm + W_ST + umma::kmaj(jrow, 32 * cg + c, 128)) = pk;
            }
#pragma unroll
            for (int c = 0; c < 32; c += 4) {
                const float4 gm = *reinterpret_cast<const float4 *>(gam + 32 * cg + c);
                const float2 lo = __fmul2_rn(make_float2(Sreg[c], Sreg[c + 1]), make_float2(gm.x, gm.y));
                const float2 hi = __fmul2_rn(make_float2(Sreg[c + 2], Sreg[c + 3]), make_float2(gm.z, gm.w));
                Sreg[c + 0] = lo.x;
                Sreg[c + 1] = lo.y;
                Sreg[c + 2] = hi.x;
                Sreg[c + 3] = hi.y;
            }
            umma::st32(tq + TM_ST + 32 * cg, Sreg);
        }
        umma::fence_proxy_async();
        umma::fence_before();
        if (__syncthreads_or(timed_out)) {
            timed_out = true;
            break;
        }

        // ------------------------------------------------------------ U~^T - S^T W^T, S^T Q~^T
        if (tid == 0) {
            umma::fence_after();
            if (has_v) {  // U~^T = V^T (T diag b)^T; V halves are 8 KB apart (LBO), k groups 1 KB (SBO)
                constexpr uint32_t id = umma::idesc_bf16(128, 64, 1, 0, 0);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    umma::mma(tmem + TM_U, umma::sdesc4(sb4 + ((W_V + b * 16384 + ks * 2048) >> 4), 8192, 1024),
                              umma::sdesc4(sb4 + ((bb + BL_TB + ks * 32) >> 4), 16, 1024), id, ks > 0 ? 1u : 0u);
            }
            constexpr uint32_t idw = umma::idesc_bf16(128, 64, 0, 1, 1);
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t kb = ks >> 2, kin = (ks & 3) * 32;
                const uint64_t a = umma::sdesc4(sb4 + ((W_ST + kb * 16384 + kin) >> 4), 16, 1024);
                umma::mma(tmem + TM_U, a, umma::sdesc4(sb4 + ((bb + BL_W + ks * 2048) >> 4), 1024, 1024), idw,
                          (has_v || ks > 0) ? 1u : 0u);
            }
            umma::commit(bar_u);
            if (save) {
                umma::bulk_store(P.save_s + ((size_t)(sbase + j) * H + h) * 32768u, sb + W_ST, 32768u);
                umma::bulk_commit();
            }
            if (need_q) {
                constexpr uint32_t idq = umma::idesc_bf16(128, 64, 0, 0, 0);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    const uint32_t kb = ks >> 2, kin = (ks & 3) * 32;
                    umma::mma(tmem + TM_O, umma::sdesc4(sb4 + ((W_ST + kb * 16384 + kin) >> 4), 16, 1024),
                              umma::sdesc4(sb4 + ((bb + BL_QT + kb * 8192 + kin) >> 4), 16, 1024), idq,
                              ks > 0 ? 1u : 0u);
                }
            }
        }
        if (!umma::mbar_wait(bar_u, pm, WAIT_LIMIT)) {
            timed_out = true;
            pend_m = 0;
            pend_mph = pm;
        }
        umma::fence_after();

        // ------------------------------------------------------------ U^T (bf16) operand
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
                *reinterpret_cast<uint4 *>(sm + W_UT + umma::kmaj(jrow, 16 * cg + c, 128)) = pk;
            }
        }
        umma::fence_proxy_async();
        umma::fence_before();
        if (__syncthreads_or(timed_out)) {
            timed_out = true;
            break;
        }

        // ------------------------------------------------------------ + U^T B^T, U^T K~
        if (tid == 0) {
            umma::fence_after();
            constexpr uint32_t ido = umma::idesc_bf16(128, 64, 0, 0, 0);
            constexpr uint32_t ids = umma::idesc_bf16(128, 128, 0, 1, 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint64_t a = umma::sdesc4(sb4 + ((W_UT + ks * 32) >> 4), 16, 1024);
                if (need_q)
                    umma::mma(tmem + TM_O, a, umma::sdesc4(sb4 + ((bb + BL_BM + ks * 32) >> 4), 16, 1024), ido, 1u);
                umma::mma(tmem + TM_ST, a, umma::sdesc4(sb4 + ((bb + BL_KT + ks * 4096) >> 4), 1024, 2048), ids, 1u);
            }
            if (save) {
                // the copies of this chunk's tiles have read them before the
                // products complete (they run meanwhile), so whoever passes the
                // barrier may overwrite S^T and U^T (next chunk, output stage)
                if (P.save_u) {
                    umma::bulk_store(P.save_u + ((size_t)(sbase + j) * H + h) * 16384u, sb + W_UT, 16384u);
                    umma::bulk_commit();
                }
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
        // checkpoint: the state after token (tc + Lc) when that position of the
        // sequence is a multiple of ckpt_every (S^T lane = value column)
        // (the tensor-memory load is warp-collective: it runs whatever this
        // thread's wait returned; only the stores depend on it)
        if (p.ckpt && !transition) {
            const int rel = tc + Lc - seq0;
            const int kq = rel / p.ckpt_every - 1;
            if (rel % p.ckpt_every == 0 && kq < p.ckpt_count) {
                float *dst = p.ckpt + (((size_t)n * p.ckpt_count + kq) * H + h) * D * (size_t)dv;
                float Sreg[32];
                umma::ld32(tq + TM_ST + 32 * cg, Sreg);
                if (!timed_out) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) dst[(size_t)(32 * cg + c) * dv + vcol0 + jrow] = Sreg[c];
                }
            }
        }

        // ------------------------------------------------------------ outputs
        // staged as a row-major [64][128] bf16 tile over U^T (read by the
        // products that just completed, and in a pass that saves the tiles by
        // its copy), then written with 16-byte stores
        unsigned char *ostage = sm + W_UT;
        if (need_q) {  // staged whatever the wait returned; the barrier below decides
            float v[16];
            umma::ld16(tq + TM_O + 16 * cg, v);
#pragma unroll
            for (int tt = 0; tt < 16; ++tt)
                *reinterpret_cast<__nv_bfloat16 *>(ostage + (16 * cg + tt) * 256 + jrow * 2) =
                    __float2bfloat16_rn(p.scale * v[tt]);
        }
        umma::fence_before();
        if (__syncthreads_or(timed_out)) {
            timed_out = true;
            break;
        }
        if (need_q) {
            __nv_bfloat16 *og = reinterpret_cast<__nv_bfloat16 *>(p.o);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int idx = tid + u * NT2, t = idx >> 4, c = idx & 15;
                if (t < Lc)
                    *reinterpret_cast<uint4 *>(og + ((size_t)(tc + t) * H + h) * dv + vcol0 + c * 8) =
                        *reinterpret_cast<const uint4 *>(ostage + t * 256 + c * 16);
            }
        }
    }

    if (timed_out) {
        if (tid == 0) report_status(p.status, KDA_STATUS_TIMEOUT);
        // let a copy still in flight land and products still running finish
        // before the shared and tensor memory are released
        if (pend_b >= 0) umma::mbar_wait(bar0 + 8 * pend_b, pend_ph, WAIT_LIMIT);
        if (pend_m >= 0) umma::mbar_wait(pend_m ? bar_o : bar_u, pend_mph, WAIT_LIMIT);
    } else {
        // ------------------------------------------------------------ state out
        float *dst = nullptr;
        size_t ld_dst = (size_t)dv, col0 = (size_t)vcol0;
        if (cut_out) {
            dst = P.carry_out + ((size_t)tile * H + h) * D * D;
            ld_dst = D;
            col0 = 0;
        } else if (p.mode == MODE_SEQ) {
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
    if (save && tid == 0) umma::bulk_wait_all();  // saved tiles written before the shared memory goes
    umma::fence_before();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(tmem, 256);
}

}  // namespace sp


namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
}  // namespace

cudaError_t launch_chunk_list(const ChunkArgs &a, int units, int nslots, int2 *list, cudaStream_t st) {
    if (nslots <= 0) return cudaSuccess;
    cudaError_t e = cudaMemsetAsync(list, 0, (size_t)nslots * sizeof(int2), st);
    if (e != cudaSuccess || units <= 0) return e;
    sp::kda_chunk_list_kernel<<<units, 128, 0, st>>>(a, nslots, list);
    return cudaGetLastError();
}

namespace {
// [T][H][inner] (or [T][H] with inner = 0) tensor map with a box of box_inner x box_h x 64 tokens
bool encode_rows(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize, int inner, int H, int T,
                 int box_inner, int box_h) {
    EncodeTiledFn fn = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
    if (!fn) return false;
    const cuuint64_t Tn = (cuuint64_t)(T > 0 ? T : 1);
    cuuint32_t estr[3] = {1u, 1u, 1u};
    if (inner > 0) {
        cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)H, Tn};
        cuuint64_t strides[2] = {(cuuint64_t)inner * esize, (cuuint64_t)inner * esize * H};
        cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)box_h, 64u};
        return fn(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    cuuint64_t dims[2] = {(cuuint64_t)H, Tn};
    cuuint64_t strides[1] = {(cuuint64_t)H * esize};
    cuuint32_t box[2] = {(cuuint32_t)box_h, 64u};
    return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

cudaError_t launch_chunk_prep(const ChunkArgs &a, const int2 *list, int slot0, int slot1, unsigned char *blob,
                              bool need_q, int *claim, bool after_walk, cudaStream_t st, float *aux) {
    if (slot1 <= slot0) return cudaSuccess;
    auto kern = aux ? sp::kda_chunk_prep_aux_kernel : sp::kda_chunk_prep_kernel;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, sp::P_SMEM);
    if (e != cudaSuccess) return e;
    sp::PrepParams P;
    memset(&P, 0, sizeof(P));
    P.q = a.q;
    P.k = a.k;
    P.g = a.g;
    P.beta = a.beta;
    P.H = a.H;
    P.g_min = a.g_min;
    P.list = list;
    P.slot0 = slot0;
    P.blob = blob;
    P.need_q = (need_q && a.q) ? 1 : 0;
    P.status = a.status;
    P.nitems = (slot1 - slot0) * a.H;
    P.claim = claim;
    P.aux = aux;
    // prefetch boxes (H is a multiple of 4 for the beta box; other H prefetch nothing there)
    bool ok = encode_rows(&P.tk, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 128, a.H, a.T, 128, 1) &&
              encode_rows(&P.tg, a.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 128, a.H, a.T, 128, 1) &&
              encode_rows(&P.tq, P.need_q ? a.q : a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 128, a.H, a.T, 128, 1);
    if (ok && a.H % 4 == 0) {
        ok = encode_rows(&P.tb, a.beta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, 0, a.H, a.T, 0, 4);
        P.pf_beta = 1;
    }
    if (!ok) return cudaErrorInvalidValue;
    // persistent: two resident CTAs per SM
    static int sms = 0;
    if (sms <= 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            sms <= 0) {
            cudaGetLastError();
            sms = 152;
        }
    }
    const int grid = P.nitems < 2 * sms ? P.nitems : 2 * sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(sp::NT1);
    cfg.dynamicSmemBytes = sp::P_SMEM;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = after_walk ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, P);
}

cudaError_t launch_chunk_walk(const ChunkArgs &a, int units, const unsigned char *blob, int slot0, int slot1,
                              const float *carry_in, float *carry_out, cudaStream_t st, unsigned char *save_s,
                              unsigned char *save_u) {
    const int ntiles = (a.mode == MODE_TRANSITION) ? 2 : 1;
    if (units <= 0) return cudaSuccess;
    if (save_s && a.mode == MODE_TRANSITION) return cudaErrorInvalidValue;  // tiles are kept by state slots
    cudaError_t e = cudaFuncSetAttribute(sp::kda_chunk_walk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         sp::W_SMEM);
    if (e != cudaSuccess) return e;
    sp::WalkParams P;
    memset(&P, 0, sizeof(P));
    P.a = a;
    P.blob = blob;
    P.slot0 = slot0;
    P.slot1 = slot1;
    P.carry_in = carry_in;
    P.carry_out = carry_out;
    P.save_s = save_s;
    P.save_u = save_u;
    EncodeTiledFn fn = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
    if (!fn) return cudaErrorInvalidValue;
    const int T = a.T;
    cuuint64_t dims[3] = {(cuuint64_t)a.dv, (cuuint64_t)a.H, (cuuint64_t)(T > 0 ? T : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)a.dv * 2, (cuuint64_t)a.dv * 2 * a.H};
    cuuint32_t box[3] = {64u, 1u, 64u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    if (fn(&P.tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(a.v), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    dim3 grid(units, a.H, ntiles);
    sp::kda_chunk_walk_kernel<<<grid, sp::NT2, sp::W_SMEM, st>>>(P);
    return cudaGetLastError();
}

}  // namespace kda
