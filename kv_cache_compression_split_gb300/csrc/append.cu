// append.cu -- appending new tokens to the caches.
//
// kvc_append: copy new K/V rows into the next free slots of every unit and
// record their absolute positions (the cache keeps each generated token's K/V,
// "Rethinking KV Cache Compression" guide, §16 "KV cache 的容量公式").
//
// kvc_append_quant: KIVI ("Rethinking KV Cache Compression" guide, §2 with
// G = 32 and R = 128; §16 "4 种方法逐步执行" and "局限与最终结论").  New tokens
// enter an fp16 residual ring; every group of 32 tokens that leaves the
// residual window is quantised -- K per channel over the group's 32 tokens,
// V per token over 32-channel groups -- and packed into the block layout that
// kvc.h documents.  Quantisation decisions are exact: binary16 values are
// taken as integers in units of 2^-24, the scale is the binary16 rounding of
// the fp64 quotient (max - min) / (2^bits - 1) (the fp64 quotient of these
// operands cannot sit within fp64 rounding distance of a binary16 midpoint,
// so the two roundings equal a single correct one), and each code is the
// round-half-even integer quotient found from an fp32 estimate corrected with
// exact int64 remainders.
#include "kvc_device.cuh"
#include "kvc_internal.h"

namespace kvc {

namespace {

// ------------------------------------------------------------ slot append

__global__ void k_append_slots(int Hkv, int D, int C, int n_new, const uint4 *__restrict__ k_new,
                               const uint4 *__restrict__ v_new, uint4 *__restrict__ K,
                               uint4 *__restrict__ V, int32_t *__restrict__ pos,
                               const int32_t *__restrict__ n, const int32_t *__restrict__ seqlen,
                               int *status)
{
    const int unit = blockIdx.x;
    const int b = unit / Hkv;
    const int n0 = n[unit];
    const int T0 = seqlen[b];
    if (n0 < 0 || n0 + n_new > C) {
        if (blockIdx.y == 0 && threadIdx.x == 0)
            flag_error(status, DEV_CAPACITY);
        return;
    }
    const int cpt = D / 8; // 16-byte chunks per token row
    const long total = (long)n_new * cpt;
    for (long idx = (long)blockIdx.y * blockDim.x + threadIdx.x; idx < total;
         idx += (long)gridDim.y * blockDim.x) {
        const int t = (int)(idx / cpt), ch = (int)(idx % cpt);
        const size_t src = ((size_t)unit * n_new + t) * cpt + ch;
        const size_t dst = ((size_t)unit * C + n0 + t) * cpt + ch;
        K[dst] = k_new[src];
        V[dst] = v_new[src];
        if (ch == 0)
            pos[(size_t)unit * C + n0 + t] = T0 + t;
    }
}

// Short appends (a few tokens, the decode case): one CTA per sequence, one
// warp per KV head; after a CTA barrier thread 0 bumps the sequence's counters,
// so no second launch is needed.
__global__ void k_append_small(int Hkv, int D, int C, int n_new, const uint4 *__restrict__ k_new,
                               const uint4 *__restrict__ v_new, uint4 *__restrict__ K,
                               uint4 *__restrict__ V, int32_t *__restrict__ pos,
                               int32_t *__restrict__ n, int32_t *__restrict__ seqlen, int *status)
{
    const int b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int T0 = seqlen[b];
    const int cpt = D / 8;
    __shared__ int s_bad;
    if (threadIdx.x == 0)
        s_bad = 0;
    __syncthreads();
    for (int hk = warp; hk < Hkv; hk += nw) {
        const int unit = b * Hkv + hk;
        const int n0 = n[unit];
        if (n0 < 0 || n0 + n_new > C) {
            if (lane == 0)
                s_bad = 1;
            continue;
        }
        for (int i = lane; i < 2 * n_new * cpt; i += 32) {
            const int kv = i / (n_new * cpt), e = i % (n_new * cpt);
            const int t = e / cpt, ch = e % cpt;
            const size_t src = ((size_t)unit * n_new + t) * cpt + ch;
            const size_t dst = ((size_t)unit * C + n0 + t) * cpt + ch;
            if (kv == 0)
                K[dst] = k_new[src];
            else
                V[dst] = v_new[src];
        }
        for (int t = lane; t < n_new; t += 32)
            pos[(size_t)unit * C + n0 + t] = T0 + t;
        __syncwarp();
        if (lane == 0)
            n[unit] = n0 + n_new;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        seqlen[b] = T0 + n_new;
        if (s_bad)
            flag_error(status, DEV_CAPACITY);
    }
}

__global__ void k_append_bump(int B, int Hkv, int C, int n_new, int32_t *n, int32_t *seqlen)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < B * Hkv && n[i] >= 0 && n[i] + n_new <= C)
        n[i] += n_new;
    if (i < B)
        seqlen[i] += n_new;
}

// ------------------------------------------------------------ KIVI pack

// binary16 value times 2^24, exactly, as an integer.
__device__ __forceinline__ long long h2fix(uint16_t h)
{
    const int e = (h >> 10) & 0x1f, f = h & 0x3ff;
    const long long v = e == 0 ? (long long)f : ((long long)(f | 0x400) << (e - 1));
    return (h & 0x8000) ? -v : v;
}

struct GroupQ {
    long long zero_fix, scale_fix;
    uint16_t zero_bits, scale_bits;
};

__device__ __forceinline__ GroupQ group_params(long long mn, uint16_t mn_bits, long long mx,
                                               int bits)
{
    GroupQ q;
    q.zero_bits = (mn_bits == 0x8000) ? (uint16_t)0 : mn_bits;
    q.zero_fix = mn;
    const double quot = (double)(mx - mn) * 0x1p-24 / (double)((1 << bits) - 1);
    q.scale_bits = __half_as_ushort(__double2half(quot));
    q.scale_fix = h2fix(q.scale_bits);
    return q;
}

__device__ __forceinline__ int quant_code(long long x, const GroupQ &q, int cmax)
{
    if (q.scale_fix == 0)
        return 0;
    const long long diff = x - q.zero_fix; // >= 0
    long long c = (long long)rintf((float)diff / (float)q.scale_fix);
    const long long rem2 = 2 * (diff - c * q.scale_fix);
    if (rem2 > q.scale_fix)
        c += 1;
    else if (rem2 < -q.scale_fix)
        c -= 1;
    else if (rem2 == q.scale_fix)
        c += (c & 1);
    else if (rem2 == -q.scale_fix)
        c -= (c & 1);
    return (int)(c < 0 ? 0 : (c > cmax ? cmax : c));
}

constexpr int QTHREADS = 256;

template <int D, int BITS>
__global__ void __launch_bounds__(QTHREADS)
    k_append_quant(int Hkv, int R, int Cq, int n_new, const uint16_t *__restrict__ k_new,
                   const uint16_t *__restrict__ v_new, uint8_t *__restrict__ kb,
                   uint8_t *__restrict__ vb, uint16_t *__restrict__ k_res,
                   uint16_t *__restrict__ v_res, const int32_t *__restrict__ len, int *status)
{
    constexpr int G = KIVI_G;
    constexpr int WK = D * BITS / 32;           // u32 words per K token row
    constexpr int W = D * BITS / 128;           // words per lane-row of a V pair
    constexpr int CODE_BYTES = G * D * BITS / 8;
    constexpr int BLOCK = CODE_BYTES + 4 * D;
    constexpr int CMAX = (1 << BITS) - 1;
    constexpr int NG = D / G;                   // V channel groups per token

    __shared__ uint16_t xk[G][D];
    __shared__ uint16_t xv[G][D];
    __shared__ uint8_t ck[G][D];
    __shared__ uint8_t cv[G][D];

    const int unit = blockIdx.x;
    const int b = unit / Hkv;
    const int CR = R + G;
    const long T0 = len[b], T1 = T0 + n_new;
    auto nq = [&](long T) -> long {
        const long over = T - R;
        return over > 0 ? (over / G) * G : 0;
    };
    const long nq0 = nq(T0), nq1 = nq(T1);
    if (nq1 > Cq) {
        if (threadIdx.x == 0)
            flag_error(status, DEV_CAPACITY);
        return;
    }
    const uint16_t *kn = k_new + (size_t)unit * n_new * D;
    const uint16_t *vn = v_new + (size_t)unit * n_new * D;
    const uint16_t *kr = k_res + (size_t)unit * CR * D;
    const uint16_t *vr = v_res + (size_t)unit * CR * D;

    for (long g = nq0 / G; g < nq1 / G; ++g) {
        // gather the group's 32 tokens (ring for old tokens, input for new ones)
        for (int i = threadIdx.x; i < G * D / 8; i += QTHREADS) {
            const int t = i / (D / 8), ch = i % (D / 8);
            const long p = g * G + t;
            const uint4 *sk, *sv;
            if (p < T0) {
                const long slot = p % CR;
                sk = reinterpret_cast<const uint4 *>(kr + slot * D) + ch;
                sv = reinterpret_cast<const uint4 *>(vr + slot * D) + ch;
            } else {
                sk = reinterpret_cast<const uint4 *>(kn + (p - T0) * D) + ch;
                sv = reinterpret_cast<const uint4 *>(vn + (p - T0) * D) + ch;
            }
            reinterpret_cast<uint4 *>(&xk[t][0])[ch] = *sk;
            reinterpret_cast<uint4 *>(&xv[t][0])[ch] = *sv;
        }
        __syncthreads();

        uint8_t *kblk = kb + ((size_t)unit * (Cq / G) + g) * BLOCK;
        uint8_t *vblk = vb + ((size_t)unit * (Cq / G) + g) * BLOCK;
        uint16_t *ksz = reinterpret_cast<uint16_t *>(kblk + CODE_BYTES);
        uint16_t *vsz = reinterpret_cast<uint16_t *>(vblk + CODE_BYTES);

        // K: per channel over the group's tokens
        for (int d = threadIdx.x; d < D; d += QTHREADS) {
            long long mn = h2fix(xk[0][d]), mx = mn;
            uint16_t mnb = xk[0][d];
            for (int t = 1; t < G; ++t) {
                const long long v = h2fix(xk[t][d]);
                if (v < mn) {
                    mn = v;
                    mnb = xk[t][d];
                }
                if (v > mx)
                    mx = v;
            }
            const GroupQ q = group_params(mn, mnb, mx, BITS);
            ksz[d] = q.scale_bits;
            ksz[D + d] = q.zero_bits;
            for (int t = 0; t < G; ++t)
                ck[t][d] = (uint8_t)quant_code(h2fix(xk[t][d]), q, CMAX);
        }
        // V: per token over channel groups of 32
        for (int i = threadIdx.x; i < G * NG; i += QTHREADS) {
            const int t = i / NG, j = i % NG;
            long long mn = h2fix(xv[t][j * G]), mx = mn;
            uint16_t mnb = xv[t][j * G];
            for (int e = 1; e < G; ++e) {
                const long long v = h2fix(xv[t][j * G + e]);
                if (v < mn) {
                    mn = v;
                    mnb = xv[t][j * G + e];
                }
                if (v > mx)
                    mx = v;
            }
            const GroupQ q = group_params(mn, mnb, mx, BITS);
            vsz[j * G + t] = q.scale_bits;
            vsz[NG * G + j * G + t] = q.zero_bits;
            for (int e = 0; e < G; ++e)
                cv[t][j * G + e] = (uint8_t)quant_code(h2fix(xv[t][j * G + e]), q, CMAX);
        }
        __syncthreads();

        // pack K token rows: field i of word w holds channel (32/BITS)*w + i
        uint32_t *kw = reinterpret_cast<uint32_t *>(kblk);
        for (int i = threadIdx.x; i < G * WK; i += QTHREADS) {
            const int t = i / WK, w = i % WK;
            uint32_t word = 0;
#pragma unroll
            for (int f = 0; f < 32 / BITS; ++f)
                word |= (uint32_t)ck[t][(32 / BITS) * w + f] << (BITS * f);
            kw[i] = word;
        }
        // pack V token pairs: word ((rr + 2 pair) mod 8)*W + k, field j holds channel
        // 16*(k*(8/BITS) + j/2) + 8*(j%2) + rr; low half token 2i, high half 2i+1
        uint32_t *vw = reinterpret_cast<uint32_t *>(vblk);
        for (int i = threadIdx.x; i < (G / 2) * 8 * W; i += QTHREADS) {
            const int pair = i / (8 * W), rk = i % (8 * W), rr = rk / W, k = rk % W;
            const int slot = pair * 8 * W + ((rr + 2 * pair) & 7) * W + k;
            uint32_t word = 0;
#pragma unroll
            for (int j = 0; j < 16 / BITS; ++j) {
                const int d = 16 * (k * (8 / BITS) + j / 2) + 8 * (j % 2) + rr;
                word |= (uint32_t)cv[2 * pair][d] << (BITS * j);
                word |= (uint32_t)cv[2 * pair + 1][d] << (16 + BITS * j);
            }
            vw[slot] = word;
        }
        __syncthreads();
    }

    // residual: new tokens that stay in fp16 go to ring slot p mod (R + 32)
    const long r0 = nq1 > T0 ? nq1 : T0;
    uint4 *krw = reinterpret_cast<uint4 *>(k_res + (size_t)unit * CR * D);
    uint4 *vrw = reinterpret_cast<uint4 *>(v_res + (size_t)unit * CR * D);
    const long total = (T1 - r0) * (D / 8);
    for (long i = threadIdx.x; i < total; i += QTHREADS) {
        const long p = r0 + i / (D / 8);
        const int ch = (int)(i % (D / 8));
        const long slot = p % CR;
        krw[slot * (D / 8) + ch] = reinterpret_cast<const uint4 *>(kn + (p - T0) * D)[ch];
        vrw[slot * (D / 8) + ch] = reinterpret_cast<const uint4 *>(vn + (p - T0) * D)[ch];
    }
}

__global__ void k_len_bump(int B, int n_new, int32_t *len)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < B)
        len[i] += n_new;
}

template <int D, int BITS>
cudaError_t launch_quant_impl(const kvc_quant_cache &c, const uint16_t *k_new,
                              const uint16_t *v_new, int n_new, cudaStream_t s)
{
    k_append_quant<D, BITS><<<c.B * c.Hkv, QTHREADS, 0, s>>>(
        c.Hkv, c.R, c.Cq, n_new, k_new, v_new, c.k_blocks, c.v_blocks, c.k_res, c.v_res, c.len,
        dev_status_ptr());
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    k_len_bump<<<(c.B + 255) / 256, 256, 0, s>>>(c.B, n_new, c.len);
    return cudaGetLastError();
}

} // namespace

cudaError_t launch_append_slots(const kvc_slot_cache &c, const uint16_t *k_new,
                                const uint16_t *v_new, int n_new, cudaStream_t s)
{
    if (n_new <= 8) {
        const int warps = c.Hkv < 16 ? c.Hkv : 16;
        k_append_small<<<c.B, 32 * warps, 0, s>>>(
            c.Hkv, c.D, c.C, n_new, reinterpret_cast<const uint4 *>(k_new),
            reinterpret_cast<const uint4 *>(v_new), reinterpret_cast<uint4 *>(c.K),
            reinterpret_cast<uint4 *>(c.V), c.pos, c.n, c.seqlen, dev_status_ptr());
        return cudaGetLastError();
    }
    const int units = c.B * c.Hkv;
    const long chunks = (long)n_new * (c.D / 8);
    int gy = (int)((chunks + 255) / 256);
    if (gy > 64)
        gy = 64;
    dim3 grid(units, gy);
    k_append_slots<<<grid, 256, 0, s>>>(c.Hkv, c.D, c.C, n_new,
                                        reinterpret_cast<const uint4 *>(k_new),
                                        reinterpret_cast<const uint4 *>(v_new),
                                        reinterpret_cast<uint4 *>(c.K),
                                        reinterpret_cast<uint4 *>(c.V), c.pos, c.n, c.seqlen,
                                        dev_status_ptr());
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    const int m = units > c.B ? units : c.B;
    k_append_bump<<<(m + 255) / 256, 256, 0, s>>>(c.B, c.Hkv, c.C, n_new, c.n, c.seqlen);
    return cudaGetLastError();
}

cudaError_t launch_append_quant(const kvc_quant_cache &c, const uint16_t *k_new,
                                const uint16_t *v_new, int n_new, cudaStream_t s)
{
    if (c.D == 128)
        return c.bits == 4 ? launch_quant_impl<128, 4>(c, k_new, v_new, n_new, s)
                           : launch_quant_impl<128, 2>(c, k_new, v_new, n_new, s);
    return c.bits == 4 ? launch_quant_impl<64, 4>(c, k_new, v_new, n_new, s)
                       : launch_quant_impl<64, 2>(c, k_new, v_new, n_new, s);
}

} // namespace kvc
