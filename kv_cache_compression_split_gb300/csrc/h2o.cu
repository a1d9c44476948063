// h2o.cu -- H2O heavy-hitter scores ("Rethinking KV Cache Compression" guide,
// §2 and §16 "4 种方法逐步执行": H2O keeps the tokens with the largest
// accumulated attention; §16 "局限与最终结论": flash attention never
// materialises the probabilities, so scoring needs an extra pass).
//
// DECODE: scores[b,hk,j] += sum_{h in group(hk)} exp(logit[b,h,j] - lse[b,h])
//         from the logits / lse that the decode attention wrote.
// PREFILL, two passes over the causal prompt (tensor cores, mma.sync):
//   pass 1  per (b, h, 64 query rows): row log-sum-exp over keys j <= i
//           (online max / sum, S = Q K^T tiles, K streamed by TMA);
//   pass 2  per (b, hk, 64 keys): recompute S^T = K Q^T for every query head
//           of the group and every query tile at or below the diagonal,
//           p = 2^(s log2e scale - lse2_i), and sum p over the queries of
//           each key (fp32 per tile, fp64 across tiles).
#include "kvc_device.cuh"
#include "kvc_internal.h"

#include <math.h>

namespace kvc {

namespace {

constexpr float LOG2E = 1.4426950408889634f;

// ------------------------------------------------------------------ decode
__global__ void k_h2o_decode_acc(int Hq, int Hkv, int C, const float *__restrict__ logits,
                                 const float *__restrict__ lse, const int32_t *__restrict__ n,
                                 float *__restrict__ scores, int *status)
{
    const int unit = blockIdx.x;
    const int b = unit / Hkv, hk = unit % Hkv, g = Hq / Hkv;
    int nn = n[unit];
    if (nn > C) {
        if (blockIdx.y == 0 && threadIdx.x == 0)
            flag_error(status, DEV_CAPACITY);
        nn = C;
    }
    const int j = blockIdx.y * blockDim.x + threadIdx.x;
    if (j >= nn)
        return;
    float s = 0.f;
    for (int h = 0; h < g; ++h) {
        const size_t row = (size_t)b * Hq + hk * g + h;
        s += expf(logits[row * C + j] - lse[row]);
    }
    scores[(size_t)unit * C + j] += s;
}

// ------------------------------------------------------------------ prefill
constexpr int NCW = 4;
constexpr int NTHREADS = (NCW + 1) * 32;
constexpr int PT = 64; // rows per tile (queries in pass 1, keys in pass 2)

template <int D> struct PreCfg {
    static constexpr int NBOX = D / 64;
    static constexpr int TILE_BYTES = PT * D * 2;
    static constexpr int NSTAGE = 4;
    static constexpr int LSE_BYTES = PT * 4;
    // pass 2 stages carry the tile's lse too; stages stay 1024-byte aligned for the swizzle
    static constexpr int STAGE_BYTES = TILE_BYTES + 1024;
    static constexpr int SMEM = NSTAGE * STAGE_BYTES + 1024 + 2 * NSTAGE * 8;
};

struct PreParams {
    int Hq, Hkv, g, L, Lpad, kp_cap, C;
    const uint16_t *qp, *kp;
    float *lse2;        // [B*Hq, Lpad] row log2-sum-exp2 of scale*log2e*q.k
    float *scores;      // [B*Hkv, C]
    float scale_log2;
    int *status;
};


template <int D>
__global__ void __launch_bounds__(NTHREADS, 2)
    k_prefill_lse(const __grid_constant__ CUtensorMap tmK, const PreParams p)
{
    using Cfg = PreCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cfg::NSTAGE * Cfg::STAGE_BYTES);
    uint64_t *empty = full + Cfg::NSTAGE;

    const int nqt = (p.L + PT - 1) / PT;
    const int qt = nqt - 1 - blockIdx.y;   // heaviest query tiles first
    const int bh = blockIdx.x;              // b * Hq + h
    const int b = bh / p.Hq, h = bh % p.Hq, hk = h / p.g;
    const int unit = b * p.Hkv + hk;
    const int nkt = qt + 1;                 // causal: key tiles 0..qt
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

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
            prefetch_tmap(&tmK);
            for (int i = 0; i < nkt; ++i) {
                const int st = i % Cfg::NSTAGE;
                if (i >= Cfg::NSTAGE && !mbar_wait(&empty[st], ((i / Cfg::NSTAGE) & 1) ^ 1)) {
                    flag_error(p.status, DEV_TIMEOUT);
                    break;
                }
                uint8_t *kt = smem + st * Cfg::STAGE_BYTES;
                mbar_arrive_expect_tx(&full[st], Cfg::TILE_BYTES);
#pragma unroll
                for (int j = 0; j < Cfg::NBOX; ++j)
                    tma_load_2d(kt + j * PT * 128, &tmK, &full[st], 64 * j,
                                unit * p.kp_cap + i * PT);
            }
        }
        return;
    }

    const int r = lane >> 2, c = lane & 3, mi = lane >> 3, ri = lane & 7;
    const int q0 = qt * PT + 16 * warp;     // first query row of this warp
    // Q rows as the A operand (row-major 16 x D)
    uint32_t qa[D / 16][4];
    {
        const int ra = min(q0 + r, p.L - 1), rb = min(q0 + r + 8, p.L - 1);
        const uint32_t *qra = reinterpret_cast<const uint32_t *>(p.qp + ((size_t)bh * p.L + ra) * D);
        const uint32_t *qrb = reinterpret_cast<const uint32_t *>(p.qp + ((size_t)bh * p.L + rb) * D);
#pragma unroll
        for (int s = 0; s < D / 16; ++s) {
            qa[s][0] = qra[8 * s + c];
            qa[s][1] = qrb[8 * s + c];
            qa[s][2] = qra[8 * s + c + 4];
            qa[s][3] = qrb[8 * s + c + 4];
        }
    }
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
    const int ia = q0 + r, ib = q0 + r + 8;

    for (int i = 0; i < nkt; ++i) {
        const int st = i % Cfg::NSTAGE;
        if (!mbar_wait(&full[st], (i / Cfg::NSTAGE) & 1)) {
            flag_error(p.status, DEV_TIMEOUT);
            break;
        }
        const uint32_t kbase = smem_u32(smem + st * Cfg::STAGE_BYTES);
        float s[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
            s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
        for (int np = 0; np < 4; ++np) {
            const int krow = 16 * np + 8 * (mi >> 1) + ri;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const int ch = 2 * ks + (mi & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(swz128(kbase + (ch >> 3) * PT * 128, krow, ch & 7), b0, b1, b2, b3);
                mma16816(s[2 * np], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
                mma16816(s[2 * np + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
            }
        }
        float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const int j0 = i * PT + 8 * nt + 2 * c;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int j = j0 + e;
                s[nt][e] = (j <= ia && j < p.L) ? s[nt][e] * p.scale_log2 : -INFINITY;
                s[nt][2 + e] = (j <= ib && j < p.L) ? s[nt][2 + e] * p.scale_log2 : -INFINITY;
                mxa = fmaxf(mxa, s[nt][e]);
                mxb = fmaxf(mxb, s[nt][2 + e]);
            }
        }
        mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 1));
        mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 2));
        mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 1));
        mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 2));
        const float na = fmaxf(m_a, mxa), nb = fmaxf(m_b, mxb);
        float sa = 0.f, sb = 0.f;
        if (na != -INFINITY) {
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
                sa += ex2(s[nt][0] - na) + ex2(s[nt][1] - na);
            l_a = l_a * ex2(m_a - na) + sa;
            m_a = na;
        }
        if (nb != -INFINITY) {
#pragma unroll
            for (int nt = 0; nt < 8; ++nt)
                sb += ex2(s[nt][2] - nb) + ex2(s[nt][3] - nb);
            l_b = l_b * ex2(m_b - nb) + sb;
            m_b = nb;
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[st]);
    }
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
    if (c == 0) {
        if (ia < p.L)
            p.lse2[(size_t)bh * p.Lpad + ia] = m_a + __log2f(l_a);
        if (ib < p.L)
            p.lse2[(size_t)bh * p.Lpad + ib] = m_b + __log2f(l_b);
    }
}

template <int D>
__global__ void __launch_bounds__(NTHREADS, 2)
    k_prefill_colsum(const __grid_constant__ CUtensorMap tmQ, const PreParams p)
{
    using Cfg = PreCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cfg::NSTAGE * Cfg::STAGE_BYTES);
    uint64_t *empty = full + Cfg::NSTAGE;

    const int nt_all = (p.L + PT - 1) / PT;
    const int kt = blockIdx.y;               // key tile (tile 0 has the most query tiles)
    const int unit = blockIdx.x, b = unit / p.Hkv, hk = unit % p.Hkv;
    const int nq_tiles = nt_all - kt;         // query tiles kt..nt_all-1
    const int nwork = p.g * nq_tiles;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

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
            prefetch_tmap(&tmQ);
            for (int i = 0; i < nwork; ++i) {
                const int st = i % Cfg::NSTAGE;
                if (i >= Cfg::NSTAGE && !mbar_wait(&empty[st], ((i / Cfg::NSTAGE) & 1) ^ 1)) {
                    flag_error(p.status, DEV_TIMEOUT);
                    break;
                }
                const int hh = i / nq_tiles, qt = kt + i % nq_tiles;
                const int bh = b * p.Hq + hk * p.g + hh;
                uint8_t *qtile = smem + st * Cfg::STAGE_BYTES;
                mbar_arrive_expect_tx(&full[st], Cfg::TILE_BYTES + Cfg::LSE_BYTES);
#pragma unroll
                for (int j = 0; j < Cfg::NBOX; ++j)
                    tma_load_2d(qtile + j * PT * 128, &tmQ, &full[st], 64 * j, bh * p.L + qt * PT);
                bulk_load(qtile + Cfg::TILE_BYTES, p.lse2 + (size_t)bh * p.Lpad + qt * PT,
                          Cfg::LSE_BYTES, &full[st]);
            }
        }
        return;
    }

    const int r = lane >> 2, c = lane & 3, mi = lane >> 3, ri = lane & 7;
    const int k0 = kt * PT + 16 * warp;       // first key of this warp
    const int ja = k0 + r, jb = k0 + r + 8;
    uint32_t ka[D / 16][4];
    {
        const int ra = min(ja, p.L - 1), rb = min(jb, p.L - 1);
        const uint32_t *kra =
            reinterpret_cast<const uint32_t *>(p.kp + ((size_t)unit * p.kp_cap + ra) * D);
        const uint32_t *krb =
            reinterpret_cast<const uint32_t *>(p.kp + ((size_t)unit * p.kp_cap + rb) * D);
#pragma unroll
        for (int s = 0; s < D / 16; ++s) {
            ka[s][0] = kra[8 * s + c];
            ka[s][1] = krb[8 * s + c];
            ka[s][2] = kra[8 * s + c + 4];
            ka[s][3] = krb[8 * s + c + 4];
        }
    }
    double acc_a = 0.0, acc_b = 0.0;

    for (int i = 0; i < nwork; ++i) {
        const int st = i % Cfg::NSTAGE;
        if (!mbar_wait(&full[st], (i / Cfg::NSTAGE) & 1)) {
            flag_error(p.status, DEV_TIMEOUT);
            break;
        }
        const int qt = kt + i % nq_tiles;
        const uint32_t qbase = smem_u32(smem + st * Cfg::STAGE_BYTES);
        const float *lse_t = reinterpret_cast<const float *>(smem + st * Cfg::STAGE_BYTES +
                                                             Cfg::TILE_BYTES);
        float s[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
            s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
        for (int np = 0; np < 4; ++np) {
            const int qrow = 16 * np + 8 * (mi >> 1) + ri;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const int ch = 2 * ks + (mi & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(swz128(qbase + (ch >> 3) * PT * 128, qrow, ch & 7), b0, b1, b2, b3);
                mma16816(s[2 * np], ka[ks][0], ka[ks][1], ka[ks][2], ka[ks][3], b0, b1);
                mma16816(s[2 * np + 1], ka[ks][0], ka[ks][1], ka[ks][2], ka[ks][3], b2, b3);
            }
        }
        float pa = 0.f, pb = 0.f;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int qi = 8 * nt + 2 * c + e;      // query within the tile
                const int iq = qt * PT + qi;
                const float l2 = lse_t[qi];
                if (iq < p.L) {
                    if (iq >= ja)
                        pa += ex2(s[nt][e] * p.scale_log2 - l2);
                    if (iq >= jb)
                        pb += ex2(s[nt][2 + e] * p.scale_log2 - l2);
                }
            }
        }
        acc_a += (double)pa;
        acc_b += (double)pb;
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[st]);
    }
    acc_a += __shfl_xor_sync(0xffffffffu, acc_a, 1);
    acc_a += __shfl_xor_sync(0xffffffffu, acc_a, 2);
    acc_b += __shfl_xor_sync(0xffffffffu, acc_b, 1);
    acc_b += __shfl_xor_sync(0xffffffffu, acc_b, 2);
    if (c == 0) {
        if (ja < p.L)
            p.scores[(size_t)unit * p.C + ja] = (float)acc_a;
        if (jb < p.L)
            p.scores[(size_t)unit * p.C + jb] = (float)acc_b;
    }
}

template <int D> cudaError_t prefill_impl(const kvc_h2o_args &a, float *lse_ws, cudaStream_t s)
{
    using Cfg = PreCfg<D>;
    static int configured = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured != dev) {
        cudaError_t e = cudaFuncSetAttribute(k_prefill_lse<D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_prefill_colsum<D>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM);
        if (e != cudaSuccess)
            return e;
        configured = dev;
    }
    PreParams p{};
    p.Hq = a.Hq;
    p.Hkv = a.Hkv;
    p.g = a.Hq / a.Hkv;
    p.L = a.L;
    p.Lpad = ((a.L + PT - 1) / PT) * PT;
    p.kp_cap = a.kp_cap;
    p.C = a.C;
    p.qp = a.qp;
    p.kp = a.kp;
    p.lse2 = lse_ws;
    p.scores = a.scores;
    const float scale = a.softmax_scale > 0.f ? a.softmax_scale : 1.0f / sqrtf((float)a.D);
    p.scale_log2 = scale * LOG2E;
    p.status = dev_status_ptr();
    CUtensorMap tk, tq;
    if (!encode_tmap_2d_f16(&tk, a.kp, D, (uint64_t)a.B * a.Hkv * a.kp_cap, 64, PT) ||
        !encode_tmap_2d_f16(&tq, a.qp, D, (uint64_t)a.B * a.Hq * a.L, 64, PT))
        return cudaErrorInvalidValue;
    const int nt = (a.L + PT - 1) / PT;
    k_prefill_lse<D><<<dim3(a.B * a.Hq, nt), NTHREADS, Cfg::SMEM, s>>>(tk, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    k_prefill_colsum<D><<<dim3(a.B * a.Hkv, nt), NTHREADS, Cfg::SMEM, s>>>(tq, p);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_h2o_decode_acc(const kvc_h2o_args &a, cudaStream_t s)
{
    dim3 grid(a.B * a.Hkv, (a.C + 255) / 256);
    k_h2o_decode_acc<<<grid, 256, 0, s>>>(a.Hq, a.Hkv, a.C, a.logits, a.lse, a.n, a.scores,
                                          dev_status_ptr());
    return cudaGetLastError();
}

cudaError_t launch_h2o_prefill(const kvc_h2o_args &a, float *lse_ws, cudaStream_t s)
{
    return a.D == 128 ? prefill_impl<128>(a, lse_ws, s) : prefill_impl<64>(a, lse_ws, s);
}

} // namespace kvc
