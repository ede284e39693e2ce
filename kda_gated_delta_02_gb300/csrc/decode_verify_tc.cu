// decode_verify_tc.cu -- fused speculative-decode verify with replay on the
// sm_103a tensor cores (tcgen05.mma, accumulators in tensor memory), dk = dv = 128.
//
// "Noyaux d'inference", section 1 "Le decodage KDA": only the projected inputs
// of draft tokens are cached; the accepted prefix is replayed on chip, and one
// kernel runs short conv -> input norm -> gating -> recurrence -> output norm
// over the replayed tokens, the bonus token and the next draft window, writing
// back the state reached after the bonus token.
//
// One CTA (8 warps; thread (c, half) = channel c, tokens 8 half .. 8 half + 7)
// owns one (request, head).  The a + 1 + Wd <= 16 tokens form one tile and the
// recurrence over it is the chunk (WY) form on that tile, with per-channel
// running decays x_t = prod_{r<=t} e^{g_r} from the window start:
//   QX = q^ . x, KX = k^ . x, KR = k^ / x,  K~_s = k^_s . x_a / x_s (s <= a)
//   A[t,s] = b_t KX_t . KR_s (s < t),  B[t,s] = QX_t . KR_s (s <= t)
//   T = (I + A)^{-1},  U = T diag(b) (V - KX S0)
//   O = scale (QX S0 + B U) -> RMSNorm over dv,  S_a = Diag(x_a) S0 + K~^T U
// (U = T diag(b) V - W S0 with W = T diag(b) KX, regrouped so that the only
// products with S0 are the two 16-row ones.)  Products run transposed with
// dv (or dk) on the MMA's M = 128:
//   batch 1   D[j][QX|KX rows]  = S0^T [QX hi|lo ; KX hi|lo]^T      (N = 64, K = dk)
//             D[QX|KX rows][s]  = [QX hi|lo ; KX hi|lo] [KR hi|lo]^T (N = 32, K = dk)
//   then      U = T diag(b) P, P = V - KX S0, as the fp32 forward substitution
//             (I + A) U = diag(b) P, one value column per thread (no T formed)
//   batch 2   S = K~^T U                                             (N = 128, K = 16)
// and O = QX S0 + B U on the CUDA cores in fp32 while batch 2 runs.
// Operands derived on chip (QX, KX, KR, K~, U) are split into
// bf16 hi + lo parts and multiplied as hi*hi + hi*lo + lo*hi, which keeps
// about 16 mantissa bits; the state is read once as bf16 (exact as an MMA
// operand) and written back rounded once (nearest even).  The state tile moves
// between HBM and shared memory by TMA in the 128-byte swizzled layout, which
// is also the MN-major operand layout of S0^T.
#include <cuda.h>  // CUtensorMap
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "kda_common.cuh"
#include "kda_internal.h"
#include "kda_umma.cuh"

namespace kda {
namespace vtc {

constexpr int D = 128, VT = 16, NT = 256, HT = 8, NR = HT + 3;

// shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_S0 = 0;       // state bf16 [dk][dv]: two 64-wide swizzled halves [128][128 B]
constexpr uint32_t OFF_X = 32768;    // [QX hi | QX lo | KX hi | KX lo]: MN-major, row = key channel, 64 columns
constexpr uint32_t OFF_KR = 49152;   // KR hi, KR lo: K-major 32 rows x dk; from here on 16 KB are also
                                     // the rows 64..127 that the M = 128 product over X reads (discarded)
constexpr uint32_t OFF_RAW = OFF_X;  // before the operands: pre-conv rows [<= 18][q|k|v][128] bf16
constexpr uint32_t OFF_GR = OFF_X + 18 * 768;  //   and g rows [<= 15][128] bf16, up to 50432
constexpr uint32_t OFF_PF = OFF_X;           // after batch 1: P = V - KX S0, fp32 [16][128]
constexpr uint32_t OFF_UF = OFF_X + 8192;    //   U, fp32 [16][128]
constexpr uint32_t OFF_AF = 54272;   //   A fp32 [16][16] (strictly lower)
constexpr uint32_t OFF_BF = 55360;   //   B fp32 [16][16] (masked)
constexpr uint32_t OFF_P = 57344;    // 128 rows; k 0-31: K~^T (hi 0-15, lo 16-31), k 32-63: U^T (hi, lo)
constexpr uint32_t OFF_BETA = 73728; // fp32 [16]
constexpr uint32_t OFF_RN = 73792;   // fp32 [32]: 1/||q_t||, 1/||k_t||
constexpr uint32_t OFF_XA = 73920;   // fp32 [128]: x_a per key channel
constexpr uint32_t OFF_CAR = 74432;  // fp32 [128]: x_7 per channel (decay carried to tokens 8-15)
constexpr uint32_t OFF_PART = 74944; // fp32 [8][16] per-warp partial sums (input norms)
constexpr uint32_t OFF_PART2 = 75456;// fp32 [8][8] per-warp partial sums (output norm)
constexpr uint32_t OFF_BAR = 75712;  // 5 mbarriers: state tile, MMA batch 1, (spare), MMA batch 2, rows
constexpr uint32_t OFF_TMEM = 75752; // tensor-memory base address
constexpr uint32_t SMEM_BYTES = 75760 + 1024;  // + alignment slack; three CTAs fit one SM

// tensor-memory columns (128 allocated)
constexpr uint32_t TM_Q = 0;    // S0^T QX^T: hi tokens in columns 0-15, lo in 16-31
constexpr uint32_t TM_K = 32;   // S0^T KX^T: hi 32-47, lo 48-63
constexpr uint32_t TM_AB = 64;  // X KR^T, lanes 0-63 (32 columns)
constexpr uint32_t TM_S = 0;    // K~^T U (128 columns, batch 3, after all of the above are read)
constexpr uint32_t TMEM_COLS = 128;
constexpr uint32_t WAIT_LIMIT = 1u << 24;
// The bound of thread 0's wait for the first batch of products.  A test build
// (KDA_TEST_SHORT_FIRST_WAIT) gives up on it at once, to exercise the timeout
// path: status reported, the copies and the products still in flight drained
// (full bound), tensor memory freed.  The library itself uses the full bound.
#ifdef KDA_TEST_SHORT_FIRST_WAIT
constexpr uint32_t FIRST_WAIT_LIMIT = 0;
#else
constexpr uint32_t FIRST_WAIT_LIMIT = WAIT_LIMIT;
#endif

struct VtcParams {
    VerifyArgs a;
    CUtensorMap ts;            // state [R*H][dk][dv] bf16, box 64 x 128 x 1, 128-byte swizzle
    CUtensorMap tt, tc, tn;    // tail / cached / new q|k|v rows as [rows][3][H][128], box 128 x 1 x 3 x n
    CUtensorMap tgc, tgn;      // cached / new g rows as [rows][H][128], box 128 x 1 x n
};

__device__ __forceinline__ float bf2f(uint16_t u) { return __uint_as_float((uint32_t)u << 16); }
// hi / lo parts of two values, each pair packed as bf16x2 (a in the low
// half): the roundings of two scalar splits, by packed conversions
__device__ __forceinline__ void split_pair(float a, float b, uint32_t &hi, uint32_t &lo) {
    hi = pack_bf16(a, b);
    const float2 h = unpack_bf16(hi);
    lo = pack_bf16(a - h.x, b - h.y);
}
// hi / lo parts of 8 consecutive values packed as 4 x bf16x2 each
__device__ __forceinline__ void split8(const float *x, uint32_t (&hi)[4], uint32_t (&lo)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) split_pair(x[2 * i], x[2 * i + 1], hi[i], lo[i]);
}
// One row of a K-major 128-byte swizzled tile: 16-byte chunk j (elements
// 8j .. 8j+7 of the row's first 64) sits at chunk j ^ (row & 7).
__device__ __forceinline__ uint32_t chunk_addr(uint32_t row_base, int row, int j) {
    return row_base + (uint32_t)(((j ^ (row & 7)) & 7) << 4);
}
// 8 values as the hi chunk j and the lo chunk j + 2 of a swizzled row
__device__ __forceinline__ void store_split8(uint32_t row_base, int row, int j, const float *x) {
    uint32_t hi[4], lo[4];
    split8(x, hi, lo);
    sts128(chunk_addr(row_base, row, j), hi[0], hi[1], hi[2], hi[3]);
    sts128(chunk_addr(row_base, row, j + 2), lo[0], lo[1], lo[2], lo[3]);
}

// Transpose-reduce over the warp: N (32, 16 or 8) values per lane in; entry
// (lane * N / 32) summed over all 32 lanes comes out in every lane that
// holds that entry.
template <int N>
__device__ __forceinline__ float warp_transpose_sum(float (&v)[N], int lane) {
#pragma unroll
    for (int n = N, o = 16; n > 1; n >>= 1, o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = up ? v[i] : v[i + n / 2];
            const float keep = up ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    float x = v[0];
#pragma unroll
    for (int o = 32 / N / 2; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__global__ void __launch_bounds__(NT, 3) kda_verify_tc_kernel(const __grid_constant__ VtcParams P) {
    const VerifyArgs &p = P.a;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(sm);
    const uint32_t sb4 = sb >> 4;
    float *sAf = reinterpret_cast<float *>(sm + OFF_AF);
    float *sPf = reinterpret_cast<float *>(sm + OFF_PF);
    float *sUf = reinterpret_cast<float *>(sm + OFF_UF);
    float *sBf = reinterpret_cast<float *>(sm + OFF_BF);
    float *sBeta = reinterpret_cast<float *>(sm + OFF_BETA);
    float *sRN = reinterpret_cast<float *>(sm + OFF_RN);
    float *sXa = reinterpret_cast<float *>(sm + OFF_XA);
    float *sCar = reinterpret_cast<float *>(sm + OFF_CAR);
    float *sPart = reinterpret_cast<float *>(sm + OFF_PART);
    float *sPart2 = reinterpret_cast<float *>(sm + OFF_PART2);
    const uint32_t bar0 = sb + OFF_BAR;  // state tile
    uint32_t *sTmem = reinterpret_cast<uint32_t *>(sm + OFF_TMEM);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // thread (c, hf): channel c of q, k, v (TMEM lane c), tokens 8 hf .. 8 hf + 7
    const int c = tid & (D - 1), hf = tid >> 7, t0 = HT * hf;
    const int H = p.H, W = p.W, Wd = p.Wd;
    const int unit = blockIdx.x;
    const int h = unit % H, r = unit / H;
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
    const int ntok = a + 1 + dr;  // <= 15 (host-checked Wd <= 7), so a <= 7 lies in the first half
    const size_t HD = (size_t)H * D, Cq = 3 * HD;
    const size_t chq = (size_t)h * D + c;

    // ---------------------------------------------------------------- setup, loads
    // One thread starts every copy of the unit: the state tile by TMA, and the
    // window's pre-conv q|k|v rows of this head and its g rows as whole boxes
    // (tail rows, all Wd cached rows, the Wd + 1 new rows) into the row region:
    // window row pr sits at row region pr when pr < W-1+a, else pr + Wd - a
    // (cached rows a .. Wd-1 are copied but not used).
    const uint32_t bar_raw = bar0 + 32;
    if (tid == 0) {
        for (int b = 0; b < 5; ++b) umma::mbar_init(bar0 + 8 * b, b == 1 ? 2u : 1u);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        umma::mbar_expect_tx(bar0, 32768u);
        umma::tma_load_3d(sb + OFF_S0, &P.ts, 0, 0, unit, bar0);
        umma::tma_load_3d(sb + OFF_S0 + 16384, &P.ts, 64, 0, unit, bar0);
        umma::mbar_expect_tx(bar_raw, (uint32_t)(W - 1 + 2 * Wd + 1) * 768u + (uint32_t)(2 * Wd + 1) * 256u);
        if (W > 1) umma::tma_load_4d(sb + OFF_RAW, &P.tt, 0, h, 0, r * (W - 1), bar_raw);
        if (Wd > 0) {
            umma::tma_load_4d(sb + OFF_RAW + (uint32_t)(W - 1) * 768u, &P.tc, 0, h, 0, r * Wd, bar_raw);
            umma::tma_load_3d(sb + OFF_GR, &P.tgc, 0, h, r * Wd, bar_raw);
        }
        umma::tma_load_4d(sb + OFF_RAW + (uint32_t)(W - 1 + Wd) * 768u, &P.tn, 0, h, 0, r * (Wd + 1), bar_raw);
        umma::tma_load_3d(sb + OFF_GR + (uint32_t)Wd * 256u, &P.tgn, 0, h, r * (Wd + 1), bar_raw);
    }
    if (warp == 0) umma::tmem_alloc(sb + OFF_TMEM, TMEM_COLS);
    float braw = 0.f;
    if (tid < ntok) {
        const uint16_t *src = (tid < a) ? reinterpret_cast<const uint16_t *>(p.cached_b) + ((size_t)r * Wd + tid) * H
                                        : reinterpret_cast<const uint16_t *>(p.new_b) + ((size_t)r * (Wd + 1) + (tid - a)) * H;
        braw = bf2f(src[h]);
    }
    float wq[4], wk[4], wv[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        wq[j] = (j < W) ? p.conv_w[chq * W + j] : 0.f;
        wk[j] = (j < W) ? p.conv_w[(HD + chq) * W + j] : 0.f;
        wv[j] = (j < W) ? p.conv_w[(2 * HD + chq) * W + j] : 0.f;
    }
    bool ok = true;
    if (tid == 0) ok = umma::mbar_wait(bar_raw, 0, WAIT_LIMIT);
    ok = __syncthreads_and(ok) != 0;  // the rows are in (and the barriers initialised)

    // pre-conv window rows t0 .. t0 + 10 of channel c (row i is token i - (W - 1));
    // rows past the last token were not copied and are never used
    uint16_t rq[NR], rk[NR], rv[NR], gr[HT];
    {
        const int split = W - 1 + a, shift = Wd - a;  // new rows sit shift rows further on
        const uint32_t rb = sb + OFF_RAW + (uint32_t)c * 2u;
#pragma unroll
        for (int i = 0; i < NR; ++i) {
            const int pr = t0 + i;
            const uint32_t ad = rb + (uint32_t)(pr + (pr >= split ? shift : 0)) * 768u;
            rq[i] = lds16(ad);
            rk[i] = lds16(ad + 256u);
            rv[i] = lds16(ad + 512u);
        }
        const uint32_t gb = sb + OFF_GR + (uint32_t)c * 2u;
#pragma unroll
        for (int j = 0; j < HT; ++j) {
            const int t = t0 + j;
            gr[j] = lds16(gb + (uint32_t)(t + (t >= a ? shift : 0)) * 256u);
        }
    }
    // conv tail write-back: the W-1 most recent pre-conv rows up to the bonus
    // token (window rows a+1 .. a+W-1), this head's q|k|v pieces, bitwise, as
    // 16-byte copies from the row region; every tail row was read above
    if (ok && tid < 48 * (W - 1)) {
        const int m = tid / 48, rem = tid - 48 * m, part = rem >> 4, q = rem & 15;
        const int pr = a + 1 + m, row = pr + (pr >= W - 1 + a ? Wd - a : 0);
        const uint4 v = lds128(sb + OFF_RAW + (uint32_t)row * 768u + (uint32_t)part * 256u + 16u * q);
        *reinterpret_cast<uint4 *>(reinterpret_cast<unsigned char *>(p.tail) +
                                   (((size_t)r * (W - 1) + m) * Cq + (size_t)part * HD + (size_t)h * D) * 2 + 16 * q) = v;
    }

    // ---------------------------------------------------------------- conv, gates
    const bool silu = p.conv_act == KDA_CONV_SILU;
    float yq[HT], yk[HT], yv[HT];
#pragma unroll
    for (int j = 0; j < HT; j += 2) {
        // the taps as packed f32x2 fused multiply-adds (each lane rounds like
        // fmaf): q and k of one token, v of two
        float2 sqk0 = make_float2(0.f, 0.f), sqk1 = sqk0, sv2 = sqk0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (i < W) {
                sqk0 = __ffma2_rn(make_float2(wq[i], wk[i]), make_float2(bf2f(rq[j + i]), bf2f(rk[j + i])), sqk0);
                sqk1 = __ffma2_rn(make_float2(wq[i], wk[i]), make_float2(bf2f(rq[j + 1 + i]), bf2f(rk[j + 1 + i])),
                                  sqk1);
                sv2 = __ffma2_rn(make_float2(wv[i], wv[i]), make_float2(bf2f(rv[j + i]), bf2f(rv[j + 1 + i])), sv2);
            }
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            float sq = u ? sqk1.x : sqk0.x, sk = u ? sqk1.y : sqk0.y, sv = u ? sv2.y : sv2.x;
            if (silu) {  // y / (1 + e^{-y}); the fast quotient is 0 where e^{-y} overflows, the limit
                sq = __fdividef(sq, 1.f + __expf(-sq));
                sk = __fdividef(sk, 1.f + __expf(-sk));
                sv = __fdividef(sv, 1.f + __expf(-sv));
            }
            const bool live = t0 + j + u < ntok;
            yq[j + u] = live ? sq : 0.f;
            yk[j + u] = live ? sk : 0.f;
            yv[j + u] = live ? sv : 0.f;
        }
    }
    // decay x_t = prod_{r<=t} e^{max(-softplus(g_r), g_min)}; e^{-softplus(g)}
    // is 1 / (1 + e^g), and the floor commutes with the exponential.  The
    // second half's products are completed with x_7 after the next barrier.
    float xd[HT];
    {
        const float emin = __expf(p.g_min);
        float run = 1.f;
#pragma unroll
        for (int j = 0; j < HT; ++j) {
            if (t0 + j < ntok) run *= fmaxf(__fdividef(1.f, 1.f + __expf(bf2f(gr[j]))), emin);
            xd[j] = run;
        }
        if (hf == 0) {
            sCar[c] = run;
            float xa0 = run;
#pragma unroll
            for (int j = 0; j < HT; ++j)
                if (j == a) xa0 = xd[j];
            sXa[c] = xa0;
        }
    }
    if (tid < VT) sBeta[tid] = (tid < ntok) ? 1.f / (1.f + __expf(-braw)) : 0.f;

    // input norms: per-token sums of squares over the D channels
    {
        float v[16];
#pragma unroll
        for (int j = 0; j < HT; ++j) {
            const float2 sq2 = __fmul2_rn(make_float2(yq[j], yk[j]), make_float2(yq[j], yk[j]));
            v[j] = sq2.x;
            v[HT + j] = sq2.y;
        }
        const float s = warp_transpose_sum<16>(v, lane);
        if ((lane & 1) == 0) sPart[warp * 16 + (lane >> 1)] = s;
    }
    __syncthreads();
    if (tid < 32) {  // entry tid = (q|k, token): the four warps of that token's half
        const int t = tid & 15, e = (tid >> 4) * HT + (t & 7), w0 = 4 * (t >> 3);
        sRN[tid] = rsqrtf(sPart[w0 * 16 + e] + sPart[(w0 + 1) * 16 + e] + sPart[(w0 + 2) * 16 + e] +
                          sPart[(w0 + 3) * 16 + e] + p.eps_in);
    }
    umma::fence_before();
    __syncthreads();
    umma::fence_after();
    const uint32_t tmem = *sTmem;
    const uint32_t tq = tmem + ((uint32_t)(32 * (warp & 3)) << 16);  // this warp's TMEM lane quadrant
    const float xa = sXa[c];
    if (hf) {
        const float car = sCar[c];
#pragma unroll
        for (int j = 0; j < HT; ++j) xd[j] *= car;
    }

    // ---------------------------------------------------------------- operands
    float kt[HT];
    {
        // X, MN-major: row c (key channel) holds the 64 columns QX hi (token t
        // at column t), QX lo (16 + t), KX hi (32 + t) and KX lo (48 + t), so
        // this thread's 8 tokens of each part are one 16-byte chunk of its row
        // (chunk 2 part + hf, swizzled by c & 7); KR stays K-major (row = token)
        const uint32_t xrow = sb + OFF_X + (uint32_t)c * 128u, cs = (uint32_t)(c & 7);
        const uint32_t rcol = sb + OFF_KR + (uint32_t)(c >> 6) * 4096u + ((uint32_t)(c & 7) << 1);
        const int ch = (c & 63) >> 3;
        const uint32_t h2 = (uint32_t)hf;
        {  // QX hi and lo
            uint32_t xh[4], xl[4];
#pragma unroll
            for (int j = 0; j < HT; j += 2)
                split_pair(yq[j] * sRN[t0 + j] * xd[j], yq[j + 1] * sRN[t0 + j + 1] * xd[j + 1], xh[j >> 1],
                           xl[j >> 1]);
            sts128(xrow + (((0u + h2) ^ cs) << 4), xh[0], xh[1], xh[2], xh[3]);
            sts128(xrow + (((2u + h2) ^ cs) << 4), xl[0], xl[1], xl[2], xl[3]);
        }
        {  // KX hi and lo; KR by token rows
            uint32_t xh[4], xl[4];
#pragma unroll
            for (int j = 0; j < HT; j += 2) {
                const int t = t0 + j;
                const float kh0 = yk[j] * sRN[VT + t], kh1 = yk[j + 1] * sRN[VT + t + 1];
                // 1 / x_t: x_t lies in [e^{16 g_min}, 1], normal in fp32, where
                // the fast quotient is within 2 ulp (the hi/lo split keeps 16 bits)
                const float rx0 = __fdividef(1.f, xd[j]), rx1 = __fdividef(1.f, xd[j + 1]);
                // rows t and t + 1 have (row & 7) == j and j + 1
                const uint32_t sw0 = (uint32_t)((ch ^ (j & 7)) << 4), sw1 = (uint32_t)((ch ^ ((j + 1) & 7)) << 4);
                split_pair(kh0 * xd[j], kh1 * xd[j + 1], xh[j >> 1], xl[j >> 1]);
                uint32_t rh, rl;
                split_pair(kh0 * rx0, kh1 * rx1, rh, rl);
                sts16(rcol + (uint32_t)t * 128u + sw0, (uint16_t)rh);
                sts16(rcol + (uint32_t)(16 + t) * 128u + sw0, (uint16_t)rl);
                sts16(rcol + (uint32_t)(t + 1) * 128u + sw1, (uint16_t)(rh >> 16));
                sts16(rcol + (uint32_t)(17 + t) * 128u + sw1, (uint16_t)(rl >> 16));
                kt[j] = (t <= a) ? kh0 * (xa * rx0) : 0.f;
                kt[j + 1] = (t + 1 <= a) ? kh1 * (xa * rx1) : 0.f;
            }
            sts128(xrow + (((4u + h2) ^ cs) << 4), xh[0], xh[1], xh[2], xh[3]);
            sts128(xrow + (((6u + h2) ^ cs) << 4), xl[0], xl[1], xl[2], xl[3]);
        }
    }
    umma::fence_proxy_async();
    __syncthreads();

    // ---------------------------------------------------------------- batch 1
    // thread 0 issues the products with S0 once its tile has landed; thread 32
    // issues X KR^T at once (two commits to one barrier of count 2)
    const bool b1 = ok;  // uniform here: thread 32's part of batch 1 is issued
    bool b2 = false;     // batch 2 issued (thread 0)
    if (tid == 0) {
        ok = umma::mbar_wait(bar0, 0, WAIT_LIMIT) && ok;
        if (ok) {
            umma::fence_after();
            constexpr uint32_t idqk = umma::idesc_bf16(128, 64, 1, 1, 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                umma::mma(tmem + TM_Q, umma::sdesc4(sb4 + ((OFF_S0 + kk * 2048) >> 4), 16384, 1024),
                          umma::sdesc4(sb4 + ((OFF_X + kk * 2048) >> 4), 1024, 1024), idqk, kk > 0 ? 1u : 0u);
            }
            umma::commit(bar0 + 8);
        }
    } else if (tid == 32 && ok) {
        umma::fence_after();
        constexpr uint32_t idab = umma::idesc_bf16(128, 32, 1, 0, 0);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t rin = (uint32_t)(kk >> 2) * 4096u + (uint32_t)(kk & 3) * 32u;
            umma::mma(tmem + TM_AB, umma::sdesc4(sb4 + ((OFF_X + kk * 2048) >> 4), 16384, 1024),
                      umma::sdesc4(sb4 + ((OFF_KR + rin) >> 4), 16, 1024), idab, kk > 0 ? 1u : 0u);
        }
        umma::commit(bar0 + 8);
    }
    // thread 0 polls the MMA barrier (both commits); a CTA barrier releases
    // the rest, so `ok` is uniform across the CTA (the TMEM loads are
    // warp-collective)
    if (tid == 0) ok = ok && umma::mbar_wait(bar0 + 8, 0, FIRST_WAIT_LIMIT);
    ok = __syncthreads_and(ok) != 0;
    umma::fence_after();

    // ---------------------------------------------------------------- A, B, T, P
    float qs[HT];
    if (ok) {
        float v0[8], v1[8];
        umma::ld8(tq + TM_Q + t0, v0);
        umma::ld8(tq + TM_Q + 16 + t0, v1);
#pragma unroll
        for (int j = 0; j < HT; j += 2) {
            const float2 q2 = __fadd2_rn(make_float2(v0[j], v0[j + 1]), make_float2(v1[j], v1[j + 1]));
            qs[j] = q2.x;
            qs[j + 1] = q2.y;
        }
        // P = V - KX S0 for value column c, tokens t0 .. t0 + 7 (fp32, for the solve)
        umma::ld8(tq + TM_K + t0, v0);
        umma::ld8(tq + TM_K + 16 + t0, v1);
#pragma unroll
        for (int j = 0; j < HT; j += 2) {
            const float2 k2 = __fadd2_rn(make_float2(v0[j], v0[j + 1]), make_float2(v1[j], v1[j + 1]));
            const float2 p2 = __fadd2_rn(make_float2(yv[j], yv[j + 1]), make_float2(-k2.x, -k2.y));
            sPf[(t0 + j) * D + c] = p2.x;
            sPf[(t0 + j + 1) * D + c] = p2.y;
        }
        // K~^T operand (k = s: hi 0-15, lo 16-31), this half's tokens
        store_split8(sb + OFF_P + (uint32_t)c * 128u, c, hf, kt);
    }
    if (ok && warp < 2) {
        // lane l holds X row 32*warp + l against KR hi (columns 0-15) and KR lo (16-31);
        // lanes 0-15 are the hi rows, lanes 16-31 the lo rows of the same tokens
        float v[32];
        umma::ld32(tq + TM_AB, v);
        float lh[VT];
#pragma unroll
        for (int s = 0; s < VT; ++s) lh[s] = __shfl_down_sync(0xffffffffu, v[s], 16);
        if (lane < VT) {
            const int t = lane;
            // warp 0: B[t][s], s <= t;  warp 1: A[t][s] = b_t KX_t . KR_s, s < t (fp32)
            const bool isA = warp == 1;
            const float bt = isA ? sBeta[t] : 1.f;
            float *dst = isA ? sAf : sBf;
#pragma unroll
            for (int s = 0; s < VT; s += 4) {
                float4 x4;
                x4.x = (isA ? (s + 0 < t) : (s + 0 <= t)) ? bt * ((v[s + 0] + v[VT + s + 0]) + lh[s + 0]) : 0.f;
                x4.y = (isA ? (s + 1 < t) : (s + 1 <= t)) ? bt * ((v[s + 1] + v[VT + s + 1]) + lh[s + 1]) : 0.f;
                x4.z = (isA ? (s + 2 < t) : (s + 2 <= t)) ? bt * ((v[s + 2] + v[VT + s + 2]) + lh[s + 2]) : 0.f;
                x4.w = (isA ? (s + 3 < t) : (s + 3 <= t)) ? bt * ((v[s + 3] + v[VT + s + 3]) + lh[s + 3]) : 0.f;
                *reinterpret_cast<float4 *>(dst + t * 16 + s) = x4;
            }
        }
    }
    ok = __syncthreads_and(ok) != 0;

    // ---------------------------------------------------------------- U by forward substitution
    // (I + A) U = diag(b) P, one value column per thread of the first half, fp32
    // (the WY form's U = T diag(b) P without forming T)
    if (ok && hf == 0) {
        float u[VT];
#pragma unroll
        for (int t = 0; t < VT; ++t) {
            float acc0 = sBeta[t] * sPf[t * D + c], acc1 = 0.f;
#pragma unroll
            for (int s4 = 0; s4 < t; s4 += 4) {
                const float4 a4 = *reinterpret_cast<const float4 *>(sAf + t * 16 + s4);
                acc0 = fmaf(-a4.x, u[s4], acc0);
                if (s4 + 1 < t) acc1 = fmaf(-a4.y, u[s4 + 1], acc1);
                if (s4 + 2 < t) acc0 = fmaf(-a4.z, u[s4 + 2], acc0);
                if (s4 + 3 < t) acc1 = fmaf(-a4.w, u[s4 + 3], acc1);
            }
            u[t] = acc0 + acc1;
        }
#pragma unroll
        for (int t = 0; t < VT; ++t) sUf[t * D + c] = u[t];
    }
    ok = __syncthreads_and(ok) != 0;
    float uu[VT];
    if (ok) {
#pragma unroll
        for (int t = 0; t < VT; ++t) uu[t] = sUf[t * D + c];
        float uh[HT];  // this half's tokens (a register select, not an indexed array)
#pragma unroll
        for (int j = 0; j < HT; ++j) uh[j] = hf ? uu[HT + j] : uu[j];
        store_split8(sb + OFF_P + (uint32_t)c * 128u, c, 4 + hf, uh);  // U^T, k = 32 + s
    }
    umma::fence_proxy_async();
    umma::fence_before();
    ok = __syncthreads_and(ok) != 0;

    // ---------------------------------------------------------------- batch 2: state
    if (tid == 0 && ok) {
        umma::fence_after();
        constexpr uint32_t ids = umma::idesc_bf16(128, 128, 0, 0, 0);
        const uint64_t kdh = umma::sdesc4(sb4 + (OFF_P >> 4), 16, 1024), kdl = umma::sdesc4(sb4 + ((OFF_P + 32) >> 4), 16, 1024);
        const uint64_t udh = umma::sdesc4(sb4 + ((OFF_P + 64) >> 4), 16, 1024);
        const uint64_t udl = umma::sdesc4(sb4 + ((OFF_P + 96) >> 4), 16, 1024);
        umma::mma(tmem + TM_S, kdh, udh, ids, 0u);
        umma::mma(tmem + TM_S, kdh, udl, ids, 1u);
        umma::mma(tmem + TM_S, kdl, udh, ids, 1u);
        umma::commit(bar0 + 24);
        b2 = true;
    }
    // outputs while the state product runs: O = scale (QX S0 + B U) in fp32
    float o[HT];
    if (ok) {
        // two tokens at a time as packed f32x2 fused multiply-adds (each lane
        // rounds like fmaf, in the same order of s)
#pragma unroll
        for (int j = 0; j < HT; j += 2) {
            const float *b0 = sBf + (t0 + j) * 16, *b1 = b0 + 16;
            float2 acc = make_float2(qs[j], qs[j + 1]);
#pragma unroll
            for (int s = 0; s < VT; s += 4) {
                const float4 x4 = *reinterpret_cast<const float4 *>(b0 + s);
                const float4 y4 = *reinterpret_cast<const float4 *>(b1 + s);
                acc = __ffma2_rn(make_float2(x4.x, y4.x), make_float2(uu[s], uu[s]), acc);
                acc = __ffma2_rn(make_float2(x4.y, y4.y), make_float2(uu[s + 1], uu[s + 1]), acc);
                acc = __ffma2_rn(make_float2(x4.z, y4.z), make_float2(uu[s + 2], uu[s + 2]), acc);
                acc = __ffma2_rn(make_float2(x4.w, y4.w), make_float2(uu[s + 3], uu[s + 3]), acc);
            }
            const float2 os = __fmul2_rn(make_float2(p.scale, p.scale), acc);
            o[j] = os.x;
            o[j + 1] = os.y;
        }
        float s2[HT];
#pragma unroll
        for (int j = 0; j < HT; j += 2) {
            const float2 o2 = __fmul2_rn(make_float2(o[j], o[j + 1]), make_float2(o[j], o[j + 1]));
            s2[j] = o2.x;
            s2[j + 1] = o2.y;
        }
        const float tot = warp_transpose_sum<8>(s2, lane);
        if ((lane & 3) == 0) sPart2[warp * 8 + (lane >> 2)] = tot;
    }
    if (tid == 0) ok = ok && umma::mbar_wait(bar0 + 24, 0, WAIT_LIMIT);
    ok = __syncthreads_and(ok) != 0;
    umma::fence_after();

    // ---------------------------------------------------------------- state write-back
    // S_a = Diag(x_a) S0 + K~^T U: row dk = c, value columns 64 hf .. 64 hf + 63,
    // written in place over S0 in the swizzled layout of the TMA store
    if (ok) {
        umma::mbar_wait(bar0, 0, WAIT_LIMIT);  // (completed long ago) orders the TMA-written tile
        const uint32_t rowb = sb + OFF_S0 + (uint32_t)hf * 16384u + (uint32_t)c * 128u;
#pragma unroll
        for (int q2 = 0; q2 < 2; ++q2) {
            float acc[32];
            umma::ld32(tq + TM_S + 64 * hf + 32 * q2, acc);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t ad = chunk_addr(rowb, c, 4 * q2 + j);
                const uint4 s0 = lds128(ad);
                const uint32_t w[4] = {s0.x, s0.y, s0.z, s0.w};
                uint32_t out[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 r2 = __ffma2_rn(make_float2(xa, xa), unpack_bf16(w[e]),
                                                 make_float2(acc[8 * j + 2 * e], acc[8 * j + 2 * e + 1]));
                    out[e] = pack_bf16(r2.x, r2.y);
                }
                sts128(ad, out[0], out[1], out[2], out[3]);
            }
        }
    }
    umma::fence_proxy_async();
    umma::fence_before();
    ok = __syncthreads_and(ok) != 0;
    if (tid == 0 && ok) {
        umma::tma_store_3d(&P.ts, 0, 0, unit, sb + OFF_S0);
        umma::tma_store_3d(&P.ts, 64, 0, unit, sb + OFF_S0 + 16384);
        umma::bulk_commit();
    }
    if (ok) {
        __nv_bfloat16 *og = reinterpret_cast<__nv_bfloat16 *>(p.o);
        const float ow = p.out_w[c];
        const int w0 = 4 * hf;
#pragma unroll
        for (int j = 0; j < HT; ++j) {
            const int t = t0 + j;
            if (t >= a && t < ntok) {
                const float tot = sPart2[w0 * 8 + j] + sPart2[(w0 + 1) * 8 + j] + sPart2[(w0 + 2) * 8 + j] +
                                  sPart2[(w0 + 3) * 8 + j];
                const float rs = rsqrtf(tot / D + p.eps_out);
                og[(((size_t)r * (Wd + 1) + (t - a)) * H + h) * D + c] = __float2bfloat16_rn(o[j] * rs * ow);
            }
        }
    } else if (tid == 0) {
        report_status(p.status, KDA_STATUS_TIMEOUT);
        umma::mbar_wait(bar_raw, 0, WAIT_LIMIT);  // let the copies land before leaving (bounded)
        umma::mbar_wait(bar0, 0, WAIT_LIMIT);
        // and the products issued finish before tensor memory is freed (when
        // this thread's own part of batch 1 was never issued the barrier stays
        // one commit short and the bounded wait outlasts thread 32's product)
        if (b1) umma::mbar_wait(bar0 + 8, 0, WAIT_LIMIT);
        if (b2) umma::mbar_wait(bar0 + 24, 0, WAIT_LIMIT);
    }
    if (warp == 0) umma::tmem_dealloc(tmem, TMEM_COLS);
    if (tid == 0 && ok) umma::bulk_wait_read();
}

}  // namespace vtc

cudaError_t launch_verify_tc(const VerifyArgs &a, cudaStream_t st) {
    typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                      const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                      CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                      CUtensorMapFloatOOBfill);
    if (a.R <= 0) return cudaSuccess;
    EncodeTiledFn fn = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
    if (!fn) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(vtc::kda_verify_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         vtc::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    vtc::VtcParams P;
    memset(&P, 0, sizeof(P));
    P.a = a;
    const size_t units = (size_t)a.R * a.H;
    cuuint64_t dims[3] = {(cuuint64_t)vtc::D, (cuuint64_t)vtc::D, (cuuint64_t)units};
    cuuint64_t strides[2] = {(cuuint64_t)vtc::D * 2, (cuuint64_t)vtc::D * vtc::D * 2};
    cuuint32_t box[3] = {64u, (cuuint32_t)vtc::D, 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    if (fn(&P.ts, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.state, dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    // q|k|v rows [rows][Cq], Cq = 3 * H * 128, seen as [rows][3][H][128]; g rows [rows][H][128]
    const cuuint64_t H = (cuuint64_t)a.H, hb = (cuuint64_t)vtc::D * 2;
    auto rows_map = [&](CUtensorMap *m, const void *base, cuuint64_t rows, cuuint32_t box_rows) {
        cuuint64_t d[4] = {(cuuint64_t)vtc::D, H, 3, rows};
        cuuint64_t st[3] = {hb, H * hb, 3 * H * hb};
        cuuint32_t bx[4] = {(cuuint32_t)vtc::D, 1u, 3u, box_rows};
        cuuint32_t es[4] = {1u, 1u, 1u, 1u};
        return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), d, st, bx, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    auto g_map = [&](CUtensorMap *m, const void *base, cuuint64_t rows, cuuint32_t box_rows) {
        cuuint64_t d[3] = {(cuuint64_t)vtc::D, H, rows};
        cuuint64_t st[2] = {hb, H * hb};
        cuuint32_t bx[3] = {(cuuint32_t)vtc::D, 1u, box_rows};
        cuuint32_t es[3] = {1u, 1u, 1u};
        return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), d, st, bx, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    const cuuint64_t R = (cuuint64_t)a.R;
    bool ok = rows_map(&P.tn, a.new_qkv, R * (a.Wd + 1), (cuuint32_t)(a.Wd + 1)) &&
              g_map(&P.tgn, a.new_g, R * (a.Wd + 1), (cuuint32_t)(a.Wd + 1));
    if (ok && a.W > 1) ok = rows_map(&P.tt, a.tail, R * (a.W - 1), (cuuint32_t)(a.W - 1));
    if (ok && a.Wd > 0)
        ok = rows_map(&P.tc, a.cached_qkv, R * a.Wd, (cuuint32_t)a.Wd) &&
             g_map(&P.tgc, a.cached_g, R * a.Wd, (cuuint32_t)a.Wd);
    if (!ok) return cudaErrorInvalidValue;
    vtc::kda_verify_tc_kernel<<<(unsigned)units, vtc::NT, vtc::SMEM_BYTES, st>>>(P);
    return cudaGetLastError();
}

}  // namespace kda
