// attend_kivi.cu -- split-KV decode attention over the quantised part of a
// KIVI cache ("Rethinking KV Cache Compression" guide, §16 "4 种方法逐步执行":
// the decode read dequantises the old cache or uses a quantised kernel).
//
// One CTA per (sequence, KV head, split); a producer lane streams the packed
// K and V group blocks of 64 tokens (two groups) into shared memory with 1-D
// bulk TMA copies; four consumer warps take 16 tokens each and never
// materialise dequantised values:
//   K (per-channel scale s_d, zero z_d per group):
//     q . k_t = sum_d (q_d s_d) c_{t,d} + sum_d q_d z_d
//     -> the scaled query q~ = q * s (fp16) is the MMA's B operand, the codes
//        c (exact small integers in fp16) are the A operand, the bias
//        sum_d q_d z_d is added to the fp32 scores.
//   V (per-token scale s_t, zero z_t per 32 channels):
//     sum_t p_t v_{t,d} = sum_t (p_t s_t) c_{t,d} + sum_t p_t z_t
//     -> p~ = p * s_t (fp16) is the B operand of O^T += C^T P~^T, and the
//        zero term is accumulated per (head, channel group) beside it.
// Codes become fp16 with the binary16 exponent trick: a field f OR-ed into
// 0x6400 (1024.0) reads as 1024 + f, and subtracting 1024 is exact.
// Results are written as split partials; the fp16 residual ring is attended
// by the slot kernel as one more partial and the combine kernel merges them.
#include "kvc_device.cuh"
#include "kvc_internal.h"

#include <math.h>

namespace kvc {

cudaError_t launch_attend_ring(int B, int Hq, int Hkv, int D, int R, const uint16_t *q,
                               const uint16_t *k_res, const uint16_t *v_res, const int32_t *len,
                               float *part_o, float *part_ml, int part_splits, int part_offset,
                               float scale, cudaStream_t s);

namespace {

constexpr int NCW = 4;
constexpr int NTHREADS = (NCW + 1) * 32;
constexpr float LOG2E = 1.4426950408889634f;

template <int D, int BITS> struct KiviCfg {
    static constexpr int G = KIVI_G;
    static constexpr int NG = D / G;                   // V channel groups
    static constexpr int WK = D * BITS / 32;           // words per K token row
    static constexpr int WPL = WK / 4;                 // K words per lane per row
    static constexpr int W = D * BITS / 128;           // V words per lane-row per pair
    static constexpr int FPW = 32 / BITS;              // fields per word
    static constexpr int HALF = FPW / 2;               // fields per 16-bit half
    static constexpr int CODE_BYTES = G * D * BITS / 8;
    static constexpr int BLOCK = CODE_BYTES + 4 * D;
    static constexpr int STAGE_BYTES = 4 * BLOCK;      // 2 K blocks + 2 V blocks
    static constexpr int NSTAGE = (BITS == 4) ? 8 : 12;
    static constexpr int SMEM = NSTAGE * STAGE_BYTES + 128 + 2 * NSTAGE * 8;
    static constexpr uint32_t MM = ((1u << BITS) - 1) | (((1u << BITS) - 1) << 16);
    static_assert(NCW * (8 * D + 16) * 4 <= NSTAGE * STAGE_BYTES, "combine scratch must fit");
};

struct KiviParams {
    int Hq, Hkv, g, Cq, R;
    int splits, tiles_per_split, part_splits;
    const uint16_t *q;
    const uint8_t *kb, *vb;
    const int32_t *len;
    float *part_o, *part_ml;
    float scale_log2;
    int *status;
};

__device__ __forceinline__ void consumer_bar()
{
    asm volatile("bar.sync 1, %0;" ::"n"(NCW * 32) : "memory");
}

__device__ __forceinline__ uint32_t hsub1024(uint32_t x)
{
    const __half2 h = *reinterpret_cast<const __half2 *>(&x);
    const __half2 r = __hsub2(h, __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400)));
    return *reinterpret_cast<const uint32_t *>(&r);
}

template <int BITS>
__device__ __forceinline__ uint32_t field_pair(uint32_t w, int j, uint32_t mm)
{
    return hsub1024(((w >> (BITS * j)) & mm) | 0x64006400u);
}

template <int D, int BITS>
__global__ void __launch_bounds__(NTHREADS, 2) k_attend_kivi(const KiviParams p)
{
    using Cfg = KiviCfg<D, BITS>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cfg::NSTAGE * Cfg::STAGE_BYTES);
    uint64_t *empty = full + Cfg::NSTAGE;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int unit = blockIdx.x / p.splits, split = blockIdx.x % p.splits;
    const int b = unit / p.Hkv, hk = unit % p.Hkv;

    const int T = p.len[b];
    const int over = T - p.R;
    int n_groups = over > 0 ? over / Cfg::G : 0;
    if (n_groups * Cfg::G > p.Cq) {
        if (threadIdx.x == 0)
            flag_error(p.status, DEV_CAPACITY);
        n_groups = p.Cq / Cfg::G;
    }
    const int unit_tiles = (n_groups + 1) / 2;
    const int tile0 = split * p.tiles_per_split;
    const int tile1 = min(unit_tiles, tile0 + p.tiles_per_split);
    const int ntiles = tile1 > tile0 ? tile1 - tile0 : 0;
    const uint8_t *kblocks = p.kb + (size_t)unit * (p.Cq / Cfg::G) * Cfg::BLOCK;
    const uint8_t *vblocks = p.vb + (size_t)unit * (p.Cq / Cfg::G) * Cfg::BLOCK;

    if (threadIdx.x == 0) {
        for (int i = 0; i < Cfg::NSTAGE; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], NCW);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == NCW) {
        if (lane == 0) {
            for (int i = 0; i < ntiles; ++i) {
                const int st = i % Cfg::NSTAGE;
                if (i >= Cfg::NSTAGE && !mbar_wait(&empty[st], ((i / Cfg::NSTAGE) & 1) ^ 1)) {
                    flag_error(p.status, DEV_TIMEOUT);
                    break;
                }
                const int g0 = 2 * (tile0 + i);
                const int ng = min(2, n_groups - g0);
                uint8_t *dst = smem + st * Cfg::STAGE_BYTES;
                mbar_arrive_expect_tx(&full[st], 2 * ng * Cfg::BLOCK);
                bulk_load(dst, kblocks + (size_t)g0 * Cfg::BLOCK, ng * Cfg::BLOCK, &full[st]);
                bulk_load(dst + 2 * Cfg::BLOCK, vblocks + (size_t)g0 * Cfg::BLOCK,
                          ng * Cfg::BLOCK, &full[st]);
            }
        }
        return;
    }

    const int r = lane >> 2, c = lane & 3;
    const int h0 = 2 * c, h1 = 2 * c + 1;
    const int gi = warp >> 1;            // group of the tile this warp works on
    const int tslice = 16 * (warp & 1);  // first token of the warp's slice in the group

    // this lane's query values (head r) over its channel range [c*D/4, (c+1)*D/4)
    float qv[D / 4];
    {
        const bool hv = r < p.g;
        const uint16_t *qrow = p.q + ((size_t)b * p.Hq + hk * p.g + (hv ? r : 0)) * D + c * (D / 4);
#pragma unroll
        for (int i = 0; i < D / 4; ++i)
            qv[i] = hv ? __half2float(__ushort_as_half(qrow[i])) : 0.f;
    }

    float acc[D / 16][4];
#pragma unroll
    for (int m = 0; m < D / 16; ++m)
        acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.f;
    float zacc[Cfg::NG];
#pragma unroll
    for (int j = 0; j < Cfg::NG; ++j)
        zacc[j] = 0.f;
    float m_run0 = -INFINITY, m_run1 = -INFINITY, l_run0 = 0.f, l_run1 = 0.f;

    for (int i = 0; i < ntiles; ++i) {
        const int st = i % Cfg::NSTAGE;
        if (!mbar_wait(&full[st], (i / Cfg::NSTAGE) & 1)) {
            flag_error(p.status, DEV_TIMEOUT);
            break;
        }
        const int g0 = 2 * (tile0 + i);
        if (g0 + gi < n_groups) {
            const uint8_t *kblk = smem + st * Cfg::STAGE_BYTES + gi * Cfg::BLOCK;
            const uint8_t *vblk = smem + st * Cfg::STAGE_BYTES + (2 + gi) * Cfg::BLOCK;
            const __half *ks = reinterpret_cast<const __half *>(kblk + Cfg::CODE_BYTES);

            // ---- q~ = q * s (B operand pairs) and bias sum_d q_d z_d for head r
            uint32_t qt[D / 8];
            float beta = 0.f;
            {
                const __half *ksl = ks + c * (D / 4);
                const __half *kzl = ks + D + c * (D / 4);
#pragma unroll
                for (int pi = 0; pi < D / 8; ++pi) {
                    const int lo = Cfg::FPW * (pi / Cfg::HALF) + (pi % Cfg::HALF);
                    const int hi = lo + Cfg::HALF;
                    qt[pi] = pack_half2(qv[lo] * __half2float(ksl[lo]),
                                        qv[hi] * __half2float(ksl[hi]));
                }
#pragma unroll
                for (int e = 0; e < D / 4; ++e)
                    beta += qv[e] * __half2float(kzl[e]);
                beta += __shfl_xor_sync(0xffffffffu, beta, 1);
                beta += __shfl_xor_sync(0xffffffffu, beta, 2);
            }
            const float beta0 = __shfl_sync(0xffffffffu, beta, 4 * h0);
            const float beta1 = __shfl_sync(0xffffffffu, beta, 4 * h1);

            // ---- S^T = C_K Q~^T over the warp's 16 tokens
            float sa[4] = {0.f, 0.f, 0.f, 0.f};
            {
                const uint32_t *kw = reinterpret_cast<const uint32_t *>(kblk);
                uint32_t wa[Cfg::WPL], wb[Cfg::WPL];
#pragma unroll
                for (int k = 0; k < Cfg::WPL; ++k) {
                    wa[k] = kw[(tslice + r) * Cfg::WK + c * Cfg::WPL + k];
                    wb[k] = kw[(tslice + r + 8) * Cfg::WK + c * Cfg::WPL + k];
                }
#pragma unroll
                for (int s = 0; s < D / 16; ++s) {
                    const int pa = 2 * s, pb = 2 * s + 1;
                    const uint32_t a0 = field_pair<BITS>(wa[pa / Cfg::HALF], pa % Cfg::HALF, Cfg::MM);
                    const uint32_t a1 = field_pair<BITS>(wb[pa / Cfg::HALF], pa % Cfg::HALF, Cfg::MM);
                    const uint32_t a2 = field_pair<BITS>(wa[pb / Cfg::HALF], pb % Cfg::HALF, Cfg::MM);
                    const uint32_t a3 = field_pair<BITS>(wb[pb / Cfg::HALF], pb % Cfg::HALF, Cfg::MM);
                    mma16816(sa, a0, a1, a2, a3, qt[pa], qt[pb]);
                }
            }
            const float x0 = (sa[0] + beta0) * p.scale_log2;
            const float x1 = (sa[1] + beta1) * p.scale_log2;
            const float x2 = (sa[2] + beta0) * p.scale_log2;
            const float x3 = (sa[3] + beta1) * p.scale_log2;
            float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            const float mn0 = fmaxf(m_run0, mx0), mn1 = fmaxf(m_run1, mx1);
            const float al0 = ex2(m_run0 - mn0), al1 = ex2(m_run1 - mn1);
            const float p0 = ex2(x0 - mn0), p2 = ex2(x2 - mn0);
            const float p1 = ex2(x1 - mn1), p3 = ex2(x3 - mn1);
            m_run0 = mn0;
            m_run1 = mn1;
            l_run0 = l_run0 * al0 + p0 + p2;
            l_run1 = l_run1 * al1 + p1 + p3;
#pragma unroll
            for (int m = 0; m < D / 16; ++m) {
                acc[m][0] *= al0;
                acc[m][1] *= al1;
                acc[m][2] *= al0;
                acc[m][3] *= al1;
            }
            // alpha of head r (the zero-term accumulator is per head r)
            const float ala = __shfl_sync(0xffffffffu, al0, r >> 1);
            const float alb = __shfl_sync(0xffffffffu, al1, r >> 1);
            const float al_r = (r & 1) ? alb : ala;

            // P^T fragments: pb0 = (p[t=2c][r], p[t=2c+1][r]), pb1 = tokens 2c+8, 2c+9
            const uint32_t pb0 = movmatrix_t(pack_half2(p0, p1));
            const uint32_t pb1 = movmatrix_t(pack_half2(p2, p3));
            const float2 pf0 = __half22float2(*reinterpret_cast<const __half2 *>(&pb0));
            const float2 pf1 = __half22float2(*reinterpret_cast<const __half2 *>(&pb1));

            // per-token V scales / zeros of this lane's four tokens
            const __half *vsz = reinterpret_cast<const __half *>(vblk + Cfg::CODE_BYTES);
            const int tk[4] = {tslice + 2 * c, tslice + 2 * c + 1, tslice + 2 * c + 8,
                               tslice + 2 * c + 9};
            const float pv[4] = {pf0.x, pf0.y, pf1.x, pf1.y};
            uint32_t ptb0[Cfg::NG], ptb1[Cfg::NG];
#pragma unroll
            for (int j = 0; j < Cfg::NG; ++j) {
                float sv[4], zv[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    sv[e] = __half2float(vsz[tk[e] * 2 * Cfg::NG + j]);
                    zv[e] = __half2float(vsz[tk[e] * 2 * Cfg::NG + Cfg::NG + j]);
                }
                ptb0[j] = pack_half2(pv[0] * sv[0], pv[1] * sv[1]);
                ptb1[j] = pack_half2(pv[2] * sv[2], pv[3] * sv[3]);
                zacc[j] = zacc[j] * al_r + pv[0] * zv[0] + pv[1] * zv[1] + pv[2] * zv[2] +
                          pv[3] * zv[3];
            }

            // ---- O^T += C_V^T P~^T per 16-channel m-tile (m-tile m lies in group m/2)
            {
                const uint32_t *vw = reinterpret_cast<const uint32_t *>(vblk);
                const int pc = 8 * (warp & 1) + c;   // token pair (2c, 2c+1) of the slice
                uint32_t wa[Cfg::W], wb[Cfg::W];
#pragma unroll
                for (int k = 0; k < Cfg::W; ++k) {
                    wa[k] = vw[pc * 2 * Cfg::WK + r * Cfg::W + k];
                    wb[k] = vw[(pc + 4) * 2 * Cfg::WK + r * Cfg::W + k];
                }
#pragma unroll
                for (int m = 0; m < D / 16; ++m) {
                    constexpr int MPW = 8 / BITS;     // m-tiles per word
                    const int k = m / MPW, jj = m % MPW;
                    const uint32_t a0 = field_pair<BITS>(wa[k], 2 * jj, Cfg::MM);
                    const uint32_t a1 = field_pair<BITS>(wa[k], 2 * jj + 1, Cfg::MM);
                    const uint32_t a2 = field_pair<BITS>(wb[k], 2 * jj, Cfg::MM);
                    const uint32_t a3 = field_pair<BITS>(wb[k], 2 * jj + 1, Cfg::MM);
                    mma16816(acc[m], a0, a1, a2, a3, ptb0[m / 2], ptb1[m / 2]);
                }
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[st]);
    }

    // ---------------- finish: zero term into O, merge the warps, write partials
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l_run0 += __shfl_xor_sync(0xffffffffu, l_run0, off);
        l_run1 += __shfl_xor_sync(0xffffffffu, l_run1, off);
    }
#pragma unroll
    for (int j = 0; j < Cfg::NG; ++j) {
        zacc[j] += __shfl_xor_sync(0xffffffffu, zacc[j], 1);
        zacc[j] += __shfl_xor_sync(0xffffffffu, zacc[j], 2);
    }
    float z0[Cfg::NG], z1[Cfg::NG];
#pragma unroll
    for (int j = 0; j < Cfg::NG; ++j) {
        z0[j] = __shfl_sync(0xffffffffu, zacc[j], 4 * h0);
        z1[j] = __shfl_sync(0xffffffffu, zacc[j], 4 * h1);
    }
#pragma unroll
    for (int m = 0; m < D / 16; ++m) {
        acc[m][0] += z0[m / 2];
        acc[m][1] += z1[m / 2];
        acc[m][2] += z0[m / 2];
        acc[m][3] += z1[m / 2];
    }
    consumer_bar();
    float *redO = reinterpret_cast<float *>(smem);
    float *redM = redO + NCW * 8 * D;
    float *redL = redM + NCW * 8;
    {
        float *w = redO + warp * 8 * D;
#pragma unroll
        for (int m = 0; m < D / 16; ++m) {
            w[h0 * D + 16 * m + r] = acc[m][0];
            w[h1 * D + 16 * m + r] = acc[m][1];
            w[h0 * D + 16 * m + r + 8] = acc[m][2];
            w[h1 * D + 16 * m + r + 8] = acc[m][3];
        }
        if (r == 0) {
            redM[warp * 8 + h0] = m_run0;
            redM[warp * 8 + h1] = m_run1;
            redL[warp * 8 + h0] = l_run0;
            redL[warp * 8 + h1] = l_run1;
        }
    }
    consumer_bar();
    for (int e = threadIdx.x; e < p.g * D; e += NCW * 32) {
        const int h = e / D, d = e % D;
        float ms = -INFINITY;
#pragma unroll
        for (int w = 0; w < NCW; ++w)
            ms = fmaxf(ms, redM[w * 8 + h]);
        float ls = 0.f, os = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
            const float mw = redM[w * 8 + h];
            const float sc = mw == -INFINITY ? 0.f : ex2(mw - ms);
            ls += sc * redL[w * 8 + h];
            os += sc * redO[(w * 8 + h) * D + d];
        }
        const size_t pi = ((size_t)unit * p.part_splits + split) * p.g + h;
        p.part_o[pi * D + d] = os;
        if (d == 0) {
            p.part_ml[2 * pi] = ls > 0.f ? ms : -INFINITY;
            p.part_ml[2 * pi + 1] = ls;
        }
    }
}

template <int D, int BITS>
cudaError_t launch_kivi_impl(const KiviParams &kp, int grid, cudaStream_t s)
{
    using Cfg = KiviCfg<D, BITS>;
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(k_attend_kivi<D, BITS>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
        if (e != cudaSuccess)
            return e;
        configured_device = dev;
    }
    k_attend_kivi<D, BITS><<<grid, NTHREADS, Cfg::SMEM, s>>>(kp);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_attend_kivi(const KiviAttendLaunch &a, cudaStream_t s)
{
    KiviParams kp{};
    kp.Hq = a.Hq;
    kp.Hkv = a.Hkv;
    kp.g = a.Hq / a.Hkv;
    kp.Cq = a.Cq;
    kp.R = a.R;
    kp.splits = a.splits;
    kp.tiles_per_split = a.tiles_per_split;
    kp.part_splits = a.splits + 1;
    kp.q = a.q;
    kp.kb = a.kb;
    kp.vb = a.vb;
    kp.len = a.len;
    kp.part_o = a.part_o;
    kp.part_ml = a.part_ml;
    kp.scale_log2 = a.scale * LOG2E;
    kp.status = dev_status_ptr();
    const int grid = a.B * a.Hkv * a.splits;
    cudaError_t e;
    if (a.D == 128)
        e = a.bits == 4 ? launch_kivi_impl<128, 4>(kp, grid, s) : launch_kivi_impl<128, 2>(kp, grid, s);
    else
        e = a.bits == 4 ? launch_kivi_impl<64, 4>(kp, grid, s) : launch_kivi_impl<64, 2>(kp, grid, s);
    if (e != cudaSuccess)
        return e;
    e = launch_attend_ring(a.B, a.Hq, a.Hkv, a.D, a.R, a.q, a.k_res, a.v_res, a.len, a.part_o,
                           a.part_ml, a.splits + 1, a.splits, a.scale, s);
    if (e != cudaSuccess)
        return e;
    return launch_combine(a.B, a.Hq, a.Hkv, a.D, a.splits + 1, a.part_o, a.part_ml, a.o, a.lse, s);
}

} // namespace kvc
