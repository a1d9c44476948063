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
                               const SlotRows rows, int *status)
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
        const long row = rows.row(unit, n0 + t);
        if (row < 0) {   // no page behind this slot
            if (ch == 0)
                flag_error(status, DEV_CAPACITY);
            continue;
        }
        const size_t dst = (size_t)row * cpt + ch;
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
                               int32_t *__restrict__ n, int32_t *__restrict__ seqlen,
                               const SlotRows rows, int *status)
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
            const long row = rows.row(unit, n0 + t);
            if (row < 0) {   // no page behind this slot
                s_bad = 1;
                continue;
            }
            const size_t dst = (size_t)row * cpt + ch;
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

// StreamingLLM decode append ("Rethinking KV Cache Compression" guide, §2 and §16
// "4 种方法逐步执行": keep the sinks and the recent window, no scores).  One token per
// sequence at position P = seqlen[b]; the token that leaves the window with this
// step, position P - n_recent - 1 (when it is not a sink), gives up its slot to the
// new token, so the cache holds exactly this step's attention window
// [0, n_sink) + [P - n_recent, P] and no eviction launch is needed.  When no slot
// holds that position (the window is not full yet) the token goes to slot n.
// One CTA per sequence, one warp per KV head: the warp scans the unit's positions
// (every load of a round in flight at once), then writes the row.
__global__ void k_stream_append(int Hkv, int D, int C, int n_sink, int n_recent,
                                const uint4 *__restrict__ k_new, const uint4 *__restrict__ v_new,
                                uint4 *__restrict__ K, uint4 *__restrict__ V,
                                int32_t *__restrict__ pos, int32_t *__restrict__ n,
                                int32_t *__restrict__ seqlen, const SlotRows rows, int *status)
{
    const int b = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int P = seqlen[b];
    const long leave = (long)P - n_recent - 1;
    const int cpt = D / 8;
    __shared__ int s_bad;
    if (threadIdx.x == 0)
        s_bad = 0;
    __syncthreads();
    for (int hk = warp; hk < Hkv; hk += nw) {
        const int unit = b * Hkv + hk;
        const int n0 = n[unit];
        if (n0 < 0 || n0 > C) {
            if (lane == 0)
                s_bad = 1;
            continue;
        }
        const int32_t *up = pos + (size_t)unit * C;
        int slot = -1;
        if (leave >= n_sink) {
            constexpr int U = 8;
            for (int base = 0; base < n0 && slot < 0; base += 32 * U) {
                int32_t pv[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int j = base + 32 * u + lane;
                    pv[u] = j < n0 ? up[j] : -1;
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const unsigned m = __ballot_sync(0xffffffffu, (long)pv[u] == leave);
                    if (m && slot < 0)
                        slot = base + 32 * u + __ffs(m) - 1;
                }
            }
        }
        const bool grow = slot < 0;
        if (grow) {
            if (n0 + 1 > C) {
                if (lane == 0)
                    s_bad = 1;
                continue;
            }
            slot = n0;
        }
        const long row = rows.row(unit, slot);
        if (row < 0) {   // no page behind this slot
            if (lane == 0)
                s_bad = 1;
            continue;
        }
        for (int i = lane; i < 2 * cpt; i += 32) {
            const size_t src = (size_t)unit * cpt + (i % cpt);
            const size_t dst = (size_t)row * cpt + (i % cpt);
            if (i < cpt)
                K[dst] = k_new[src];
            else
                V[dst] = v_new[src];
        }
        if (lane == 0) {
            pos[(size_t)unit * C + slot] = P;
            if (grow)
                n[unit] = n0 + 1;
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        seqlen[b] = P + 1;
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

// binary16 bits of the correctly rounded (to nearest, ties to even) value of
// range * 2^-24 / CMAX, for an integer 0 <= range < 2^42 and odd CMAX, in
// integer arithmetic: in units of 2^-24 binary16 has spacing 1 below 2^10
// (subnormals) and 2^k on [2^(k+10), 2^(k+11)), and its encoding k * 2^10 + m
// is continuous, so a carry of the rounded mantissa m into 2^11 lands on the
// next binade by itself.
template <int CMAX> __device__ __forceinline__ uint16_t scale_bits_rn(unsigned long long range)
{
    const unsigned long long q0 = range / CMAX;          // floor of the quotient
    if (q0 < 1024) {
        const unsigned long long r = range - q0 * CMAX;
        return (uint16_t)(q0 + (2 * r > CMAX));         // CMAX odd: no exact ties
    }
    const int k = 53 - __clzll((long long)q0);           // quotient in [2^(k+10), 2^(k+11))
    const unsigned long long div = (unsigned long long)CMAX << k;
    const unsigned long long m = q0 >> k;                 // floor(range / div)
    const unsigned long long r2 = 2 * (range - m * div);
    const unsigned long long mm = m + (r2 > div || (r2 == div && (m & 1)));
    return (uint16_t)(((unsigned long long)k << 10) + mm);
}

template <int BITS>
__device__ __forceinline__ GroupQ group_params(long long mn, uint16_t mn_bits, long long mx)
{
    GroupQ q;
    q.zero_bits = (mn_bits == 0x8000) ? (uint16_t)0 : mn_bits;
    q.zero_fix = mn;
    q.scale_bits = scale_bits_rn<(1 << BITS) - 1>((unsigned long long)(mx - mn));
    q.scale_fix = h2fix(q.scale_bits);
    return q;
}

// Code of x: round-half-even((x - zero) / scale) clamped to [0, cmax], exact.
// The estimate is formed in fp32 from the binary16 values (x - zero rounded
// once, times 1/scale), which puts it within one of the true quotient; the
// exact integer remainder (values in units of 2^-24) then decides, ties to the
// even code.  No 64-bit integer is converted to or from floating point.
__device__ __forceinline__ int quant_code_inv(uint16_t xb, long long zero_fix, float zero_f,
                                              long long scale_fix, float inv, int cmax)
{
    if (scale_fix == 0)
        return 0;
    const long long diff = h2fix(xb) - zero_fix;   // >= 0
    const float est = (__half2float(__ushort_as_half(xb)) - zero_f) * inv;
    long long c = (long long)__float2int_rn(fminf(est, 1048576.f));
    const long long rem2 = 2 * (diff - c * scale_fix);
    if (rem2 > scale_fix)
        c += 1;
    else if (rem2 < -scale_fix)
        c -= 1;
    else if (rem2 == scale_fix)
        c += (c & 1);
    else if (rem2 == -scale_fix)
        c -= (c & 1);
    return (int)(c < 0 ? 0 : (c > cmax ? cmax : c));
}

constexpr int QTHREADS = 256;

// Shared staging of one 32-token group: fp16 inputs, then codes.
template <int D> struct __align__(16) GroupSmem {
    uint16_t xk[KIVI_G][D];
    uint16_t xv[KIVI_G][D];
    uint8_t ck[KIVI_G][D];
    uint8_t cv[KIVI_G][D];
    long long zfix[2 * D];       // per K channel, then per V (token, channel group)
    long long sfix[2 * D];
    float zf[2 * D];             // zero as fp32
    float sf[2 * D];             // scale as fp32
    float inv[2 * D];            // 1 / scale (an estimate; the remainder fixes the code)
};

// Extra staging of the GEAR side data of a group's two matrices (index 0: K,
// 1: V), worked on together so that each serial step serves both.  Rows are
// padded by 8 words: 64-bit fragment loads of a half-warp (8 rows x 2 columns
// pairs) then hit every bank once.
constexpr int GM_LD = KIVI_G + 8;
template <int D> struct __align__(16) GearSmem {
    float e[2][KIVI_G][D + 8];   // residual, then R (sparse entries zeroed)
    float gm[2][KIVI_G][GM_LD];
    float gm2[2][KIVI_G][GM_LD];
    float a[2][2][KIVI_G];       // orthonormal left factors
    int hist[3][2][256];         // radix digit counts, three buffers in rotation
    int scan[2][QTHREADS / 32];
    int red[2][QTHREADS / 32];
};

__device__ __forceinline__ uint32_t h2_bits(__half2 h)
{
    return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ __half2 bits_h2(uint32_t u)
{
    return *reinterpret_cast<const __half2 *>(&u);
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// One 16 x 8 tile C[i][j] = sum_k X[i0 + i][k] Y[j0 + j][k] of fp32 row-major matrices
// in shared memory (leading dimension LD), with tensor cores: sc * X and sc * Y are
// split into binary16 high and low parts and C = Xh Yh^T + Xh Yl^T + Xl Yh^T (fp32
// accumulation; each product carries a relative error of about 2^-22, and sc keeps the
// values in binary16's normal range).  One warp; fragment layout of mma m16n8k16.
__device__ __forceinline__ void split_h2(float x, float y, uint32_t &hi, uint32_t &lo)
{
    const __half2 h = __floats2half2_rn(x, y);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(x - hf.x, y - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

template <int K, int LD>
__device__ __forceinline__ void xyt_tile(const float *X, int i0, const float *Y, int j0,
                                         float sc, float (&c)[4])
{
    static_assert(LD % 32 == 8, "conflict-free 64-bit fragment loads need LD = 8 mod 32");
    const int lane = threadIdx.x & 31, gid = lane >> 2, tig = lane & 3;
    const float *x0 = X + (i0 + gid) * LD, *x1 = x0 + 8 * LD;
    const float *y0 = Y + (j0 + gid) * LD;
    auto ld2 = [](const float *p) { return *reinterpret_cast<const float2 *>(p); };
#pragma unroll
    for (int s = 0; s < K / 16; ++s) {
        const int k = 16 * s + 2 * tig;
        uint32_t ah[4], al[4], bh[2], bl[2];
        const float2 p0 = ld2(x0 + k), p1 = ld2(x1 + k), p2 = ld2(x0 + k + 8),
                     p3 = ld2(x1 + k + 8), q0 = ld2(y0 + k), q1 = ld2(y0 + k + 8);
        split_h2(sc * p0.x, sc * p0.y, ah[0], al[0]);
        split_h2(sc * p1.x, sc * p1.y, ah[1], al[1]);
        split_h2(sc * p2.x, sc * p2.y, ah[2], al[2]);
        split_h2(sc * p3.x, sc * p3.y, ah[3], al[3]);
        split_h2(sc * q0.x, sc * q0.y, bh[0], bl[0]);
        split_h2(sc * q1.x, sc * q1.y, bh[1], bl[1]);
        mma16816(c, ah[0], ah[1], ah[2], ah[3], bh[0], bh[1]);
        mma16816(c, ah[0], ah[1], ah[2], ah[3], bl[0], bl[1]);
        mma16816(c, al[0], al[1], al[2], al[3], bh[0], bh[1]);
    }
}

// dst = src * src for a symmetric 32 x 32 matrix (entries of magnitude <= 32), one
// 16 x 8 tile per warp (8 warps).
__device__ __forceinline__ void square32(const float (*src)[GM_LD], float (*dst)[GM_LD])
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i0 = 16 * (warp >> 2), j0 = 8 * (warp & 3), gid = lane >> 2, tig = lane & 3;
    float c[4] = {0.f, 0.f, 0.f, 0.f};
    xyt_tile<KIVI_G, GM_LD>(&src[0][0], i0, &src[0][0], j0, 1.f, c);
    dst[i0 + gid][j0 + 2 * tig] = c[0];
    dst[i0 + gid][j0 + 2 * tig + 1] = c[1];
    dst[i0 + gid + 8][j0 + 2 * tig] = c[2];
    dst[i0 + gid + 8][j0 + 2 * tig + 1] = c[3];
}

// Orthonormalise the two columns (x0, x1) a warp holds, one row per lane; a
// column with no length left becomes a unit vector orthogonal to the other.
__device__ __forceinline__ void orthonormalise2(float &x0, float &x1);

// The same with the three inner products reduced together (one round of
// shuffles): x0 / |x0| and x1 - (x0.x1 / x0.x0) x0, normalised.  Falls back to
// orthonormalise2 when |x0| vanishes or x1 loses more than 1 - 1e-3 of its
// squared length to the projection (cancellation).
__device__ __forceinline__ void orthonormalise2_fast(float &x0, float &x1)
{
    float n0 = x0 * x0, dp = x0 * x1, n1 = x1 * x1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        n0 += __shfl_xor_sync(0xffffffffu, n0, o);
        dp += __shfl_xor_sync(0xffffffffu, dp, o);
        n1 += __shfl_xor_sync(0xffffffffu, n1, o);
    }
    const float rest = n1 - dp * dp / n0;
    if (!(n0 > 1e-30f) || !(rest > 1e-3f * n1) || !(n1 > 1e-24f)) {
        orthonormalise2(x0, x1);
        return;
    }
    const float f = dp / n0;
    x1 = (x1 - f * x0) * rsqrtf(rest);
    x0 *= rsqrtf(n0);
}

__device__ __forceinline__ void orthonormalise2(float &x0, float &x1)
{
    const int lane = threadIdx.x & 31;
    float n0 = warp_sum(x0 * x0);
    if (n0 > 1e-30f)
        x0 *= rsqrtf(n0);
    else
        x0 = lane == 0 ? 1.f : 0.f;
    x1 -= warp_sum(x0 * x1) * x0;
    float n1 = warp_sum(x1 * x1);
    if (!(n1 > 1e-24f)) {
        const float x0_first = __shfl_sync(0xffffffffu, x0, 0);
        x1 = lane == (fabsf(x0_first) > 0.7f ? 1 : 0) ? 1.f : 0.f;
        x1 -= warp_sum(x0 * x1) * x0;
        n1 = warp_sum(x1 * x1);
    }
    x1 *= rsqrtf(n1);
}

// Digit of the radix select over one matrix's keys, found by every warp from
// the same histogram h (no barrier needed to share it): lane L reads digits
// 255 - 8L - k (k = 0..7, descending); the digit is the first one from the top
// whose cumulative count reaches `need`, and `need` becomes the rank left
// within it.  With fewer matching keys than needed (cannot happen for
// consistent input) the digit is 0, as a downward scan would end.
__device__ __forceinline__ void radix_digit(const int *h_all, int &digit, int &need)
{
    const int lane = threadIdx.x & 31;
    int h[8], tot = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        h[k] = h_all[255 - 8 * lane - k];
        tot += h[k];
    }
    int incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += y;
    }
    const bool mine = incl - tot < need && incl >= need;
    const unsigned any = __ballot_sync(0xffffffffu, mine);
    int dg, nd;
    if (any) {
        int cum = incl - tot, k = 0;
        for (; k < 7; ++k) {
            if (cum + h[k] >= need)
                break;
            cum += h[k];
        }
        dg = 255 - 8 * lane - k;
        nd = need - cum;
    } else {
        dg = 0;
        nd = need - (incl - h[7]);
    }
    const int src = any ? __ffs(any) - 1 : 31;
    digit = __shfl_sync(0xffffffffu, dg, src);
    need = __shfl_sync(0xffffffffu, nd, src);
}

// GEAR side blocks of both matrices of the group, written to kside (K) and
// vside (V): the residual e = fl32(x - fl32(zero + code * scale)) of every
// element, the n_s entries with the largest |e| (ties: lower flat index) as
// ascending u16 flat indices and binary16 values, and a rank-2 factorisation
// A^T B of the rest R: A [2][32] orthonormal rows spanning the dominant left
// singular subspace, B = A R; both binary16.  The subspace comes from 16 steps
// of subspace iteration on (R R^T)^4 (R R^T scaled by its largest entry, then
// squared twice), started from R R^T times a constant and a ramp.  All threads
// of the CTA; the two matrices share every barrier, and their iterations run
// in warps 0 (K) and 1 (V) at the same time.
template <int D, int BITS>
__device__ __forceinline__ void gear_sides(const GroupSmem<D> &sm, GearSmem<D> &gs,
                                           uint8_t *kside, uint8_t *vside)
{
    constexpr int G = KIVI_G, NG = D / G, N = G * D, PER = N / QTHREADS;
    constexpr int NS = (2 * G * D + 99) / 100;
    constexpr int RAW = 4 * NS + 4 * G + 4 * D;
    constexpr int SIDE = (RAW + 15) / 16 * 16;
    static_assert(QTHREADS == 256, "eight warps cover the 32 x 32 Gram matrix");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint8_t *const sides[2] = {kside, vside};
    // 1. residuals of my PER elements of each matrix: warp w owns flat indices
    //    [32 PER w, 32 PER (w + 1)), lane L of it 32 u + L (u < PER), so a warp's
    //    accesses cover 32 consecutive elements of one row
    const auto flat = [&](int u) { return 32 * PER * warp + 32 * u + lane; };
#pragma unroll
    for (int m = 0; m < 2; ++m) {
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const int i = flat(u), t = i / D, d = i % D;
            const int pi = m == 0 ? d : D + t * NG + d / G;
            const float x = __half2float(__ushort_as_half(m == 0 ? sm.xk[t][d] : sm.xv[t][d]));
            const float code = (float)(m == 0 ? sm.ck[t][d] : sm.cv[t][d]);
            gs.e[m][t][d] = x - fmaf(code, sm.sf[pi], sm.zf[pi]);
        }
    }
    const auto key = [&](int m, int u) {
        const int i = flat(u);
        return __float_as_uint(gs.e[m][i / D][i % D]) & 0x7fffffffu;   // bits of |e|
    };
    for (int i = tid; i < 2 * 2 * 256; i += QTHREADS)
        (&gs.hist[0][0][0])[i] = 0;
    __syncthreads();
    // 2. the NS-th largest key of each matrix: radix select, 8-bit digits from the
    //    top.  Pass p counts into buffer p mod 3 and clears buffer (p + 1) mod 3, whose
    //    last readers (pass p - 2) finished before pass p - 1's barrier.
    uint32_t prefix[2] = {0u, 0u}, mask = 0;
    int need[2] = {NS, NS};
#pragma unroll 1
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        int(*hc)[256] = gs.hist[pass % 3];
        int *hz = &gs.hist[(pass + 1) % 3][0][0];
        // histogram of the digit among keys matching the prefix; lanes with equal
        // digits add once (keys concentrate on a few exponents)
#pragma unroll
        for (int m = 0; m < 2; ++m) {
#pragma unroll
            for (int u = 0; u < PER; ++u) {
                const uint32_t k = key(m, u);
                const bool in = (k & mask) == prefix[m];
                if (!__any_sync(0xffffffffu, in))
                    continue;
                const int dg = in ? (int)((k >> shift) & 255) : 256;
                const unsigned same = __match_any_sync(0xffffffffu, dg);
                if (in && lane == __ffs(same) - 1)
                    atomicAdd(&hc[m][dg], __popc(same));
            }
        }
        if (pass < 3)
            for (int i = tid; i < 2 * 256; i += QTHREADS)
                hz[i] = 0;
        __syncthreads();
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            int dg;
            radix_digit(hc[m], dg, need[m]);
            prefix[m] |= (uint32_t)dg << shift;
        }
        mask |= 255u << shift;
    }
    // 3. keep every key above the threshold and the first `need` equal to it, in flat
    //    order: ranks from per-u ballots within the warp plus the earlier warps' totals
    const unsigned lt = (1u << lane) - 1u;
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        int wcount = 0;
#pragma unroll
        for (int u = 0; u < PER; ++u)
            wcount += __popc(__ballot_sync(0xffffffffu, key(m, u) == prefix[m]));
        if (lane == 0)
            gs.scan[m][warp] = wcount;
    }
    __syncthreads();
    uint32_t selm[2] = {0u, 0u};   // bit u: element u selected
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        int run = 0;
        for (int w = 0; w < warp; ++w)
            run += gs.scan[m][w];
        int wcount = 0;
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const uint32_t k = key(m, u);
            const unsigned tb = __ballot_sync(0xffffffffu, k == prefix[m]);
            const bool sel =
                k > prefix[m] || (((tb >> lane) & 1u) && run + __popc(tb & lt) < need[m]);
            run += __popc(tb);
            selm[m] |= (uint32_t)sel << u;
            wcount += __popc(__ballot_sync(0xffffffffu, sel));
        }
        if (lane == 0)
            gs.red[m][warp] = wcount;
    }
    __syncthreads();
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        int o = 0;
        for (int w = 0; w < warp; ++w)
            o += gs.red[m][w];
        uint16_t *idx_out = reinterpret_cast<uint16_t *>(sides[m]);
        __half *val_out = reinterpret_cast<__half *>(sides[m] + 2 * NS);
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const bool sel = (selm[m] >> u) & 1u;
            const unsigned sb = __ballot_sync(0xffffffffu, sel);
            const int pos = o + __popc(sb & lt);
            if (sel && pos < NS) {             // exactly NS are selected; the bound is a guard
                const int i = flat(u), t = i / D, d = i % D;
                idx_out[pos] = (uint16_t)i;
                val_out[pos] = __float2half_rn(gs.e[m][t][d]);
                gs.e[m][t][d] = 0.f;           // R: the rest of the residual
            }
            o += __popc(sb);
        }
    }
    __syncthreads();
    // 4. Gram matrices R R^T with tensor cores, one 16 x 8 tile of each per warp, scaled
    //    by their largest entry.  Every entry of R is at most the threshold key, so
    //    R * 2^(130 - e) (e: the threshold's exponent field) stays below 16 in binary16.
    {
        const int i0 = 16 * (warp >> 2), j0 = 8 * (warp & 3), gid = lane >> 2, tig = lane & 3;
        float c[2][4];
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const int ex = (int)((prefix[m] >> 23) & 255);
            const float sc = prefix[m] ? __int_as_float(min(257 - ex, 254) << 23) : 1.f;
            c[m][0] = c[m][1] = c[m][2] = c[m][3] = 0.f;
            xyt_tile<D, D + 8>(&gs.e[m][0][0], i0, &gs.e[m][0][0], j0, sc, c[m]);
            float mx = fmaxf(fmaxf(fabsf(c[m][0]), fabsf(c[m][1])),
                             fmaxf(fabsf(c[m][2]), fabsf(c[m][3])));
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1)
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
            if (lane == 0)
                gs.scan[m][warp] = __float_as_int(mx);
        }
        __syncthreads();
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            float mm = 0.f;
#pragma unroll
            for (int w = 0; w < QTHREADS / 32; ++w)
                mm = fmaxf(mm, __int_as_float(gs.scan[m][w]));
            const float inv_m = mm > 0.f ? 1.f / mm : 0.f;
            gs.gm[m][i0 + gid][j0 + 2 * tig] = c[m][0] * inv_m;
            gs.gm[m][i0 + gid][j0 + 2 * tig + 1] = c[m][1] * inv_m;
            gs.gm[m][i0 + gid + 8][j0 + 2 * tig] = c[m][2] * inv_m;
            gs.gm[m][i0 + gid + 8][j0 + 2 * tig + 1] = c[m][3] * inv_m;
        }
    }
    __syncthreads();
    square32(gs.gm[0], gs.gm2[0]);             // (R R^T)^2, entries <= 32
    square32(gs.gm[1], gs.gm2[1]);
    __syncthreads();
    square32(gs.gm2[0], gs.gm[0]);             // (R R^T)^4, entries <= 32^3
    square32(gs.gm2[1], gs.gm[1]);
    __syncthreads();
    // 5. dominant 2-dimensional subspaces: subspace iteration, K in warp 0 and V in
    //    warp 1, one row per lane
    if (warp < 2) {
        const int m = warp;
        float gr[G];
#pragma unroll
        for (int j = 0; j < G; ++j)
            gr[j] = gs.gm[m][lane][j];
        float x0 = 0.f, x1 = 0.f;
#pragma unroll
        for (int j = 0; j < G; ++j) {
            x0 += gr[j];
            x1 = fmaf(gr[j], (float)j - 15.5f, x1);
        }
        orthonormalise2(x0, x1);
        for (int it = 0; it < 16; ++it) {
            // y = M x, the vectors broadcast from shared memory four entries at a time
            gs.a[m][0][lane] = x0;
            gs.a[m][1][lane] = x1;
            __syncwarp();
            const float4 *a0 = reinterpret_cast<const float4 *>(gs.a[m][0]);
            const float4 *a1 = reinterpret_cast<const float4 *>(gs.a[m][1]);
            float y0 = 0.f, y1 = 0.f;
#pragma unroll
            for (int j = 0; j < G / 4; ++j) {
                const float4 u = a0[j], v = a1[j];
                y0 = fmaf(gr[4 * j], u.x, y0);
                y0 = fmaf(gr[4 * j + 1], u.y, y0);
                y0 = fmaf(gr[4 * j + 2], u.z, y0);
                y0 = fmaf(gr[4 * j + 3], u.w, y0);
                y1 = fmaf(gr[4 * j], v.x, y1);
                y1 = fmaf(gr[4 * j + 1], v.y, y1);
                y1 = fmaf(gr[4 * j + 2], v.z, y1);
                y1 = fmaf(gr[4 * j + 3], v.w, y1);
            }
            __syncwarp();
            x0 = y0;
            x1 = y1;
            orthonormalise2_fast(x0, x1);
        }
        gs.a[m][0][lane] = x0;
        gs.a[m][1][lane] = x1;
    }
    __syncthreads();
    // 6. factors: A [2][G] and B = A R [2][D], binary16; zero padding
#pragma unroll
    for (int m = 0; m < 2; ++m) {
        __half *a_out = reinterpret_cast<__half *>(sides[m] + 4 * NS);
        __half *b_out = reinterpret_cast<__half *>(sides[m] + 4 * NS + 4 * G);
        for (int i = tid; i < 2 * G; i += QTHREADS)
            a_out[i] = __float2half_rn(gs.a[m][i / G][i % G]);
        for (int i = tid; i < 2 * D; i += QTHREADS) {
            const int r = i / D, d = i % D;
            float s = 0.f;
#pragma unroll 8
            for (int t = 0; t < G; ++t)
                s = fmaf(gs.a[m][r][t], gs.e[m][t][d], s);
            b_out[i] = __float2half_rn(s);
        }
        for (int i = RAW + tid; i < SIDE; i += QTHREADS)
            sides[m][i] = 0;
    }
    __syncthreads();
}

// Quantise and pack group g of one unit (all threads of the CTA take part):
// gather its 32 tokens (old ones from the residual ring, new ones from the
// input), compute the K per-channel and V per-(token, channel-group)
// scale / zero, the codes, and write the K and V blocks.
template <int D, int BITS, bool GEAR>
__device__ __forceinline__ void pack_group(long g, long T0, int CR, const uint16_t *kn,
                                           const uint16_t *vn, const uint16_t *kr,
                                           const uint16_t *vr, uint8_t *kblk, uint8_t *vblk,
                                           GroupSmem<D> &sm, GearSmem<D> *gs, uint8_t *kside,
                                           uint8_t *vside)
{
    constexpr int G = KIVI_G;
    constexpr int WK = D * BITS / 32;           // u32 words per K token row
    constexpr int W = D * BITS / 128;           // words per lane-row of a V pair
    constexpr int CODE_BYTES = G * D * BITS / 8;
    constexpr int CMAX = (1 << BITS) - 1;
    constexpr int NG = D / G;                   // V channel groups per token
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
        reinterpret_cast<uint4 *>(&sm.xk[t][0])[ch] = *sk;
        reinterpret_cast<uint4 *>(&sm.xv[t][0])[ch] = *sv;
    }
    __syncthreads();
    uint16_t *ksz = reinterpret_cast<uint16_t *>(kblk + CODE_BYTES);
    uint16_t *vsz = reinterpret_cast<uint16_t *>(vblk + CODE_BYTES);
    // 1. parameters, one set per thread: sets [0, D) are the K channels (over the
    //    group's 32 tokens), sets [D, 2D) the V (token, 32-channel group) pairs.
    //    The extremes are taken on binary16 pairs: min and max of binary16 values
    //    are exact and do not depend on the scan order (a -0 / +0 tie is harmless:
    //    a -0 zero point is stored as +0, and both are 0 in fixed point).  K: the
    //    threads 2p and 2p + 1 scan channels 2p, 2p + 1 over tokens [0, 16) and
    //    [16, 32) and swap their partial extremes; thread 2p + c keeps channel
    //    2p + c.  V: a thread reads its set's 32 contiguous values as four 16-byte
    //    chunks, starting at a chunk rotated by (token, group) so that a warp's
    //    loads spread over all banks.
    static_assert(2 * D <= QTHREADS, "one parameter set per thread");
    if (threadIdx.x < 2 * D) {
        const int i = threadIdx.x;
        uint16_t mnb, mxb;
        if (i < D) {
            const int pr = i >> 1, c = i & 1;
            const __half2 *col = reinterpret_cast<const __half2 *>(&sm.xk[16 * c][2 * pr]);
            __half2 mn2 = col[0], mx2 = mn2;
#pragma unroll
            for (int e = 1; e < G / 2; ++e) {
                const __half2 v = col[e * (D / 2)];
                mn2 = __hmin2(mn2, v);
                mx2 = __hmax2(mx2, v);
            }
            const uint32_t omn = __shfl_xor_sync(0xffffffffu, h2_bits(mn2), 1);
            const uint32_t omx = __shfl_xor_sync(0xffffffffu, h2_bits(mx2), 1);
            const uint32_t a = h2_bits(__hmin2(mn2, bits_h2(omn)));
            const uint32_t b = h2_bits(__hmax2(mx2, bits_h2(omx)));
            mnb = (uint16_t)(c ? a >> 16 : a & 0xffffu);
            mxb = (uint16_t)(c ? b >> 16 : b & 0xffffu);
        } else {
            const int a = i - D, t = a / NG, j = a % NG;
            const uint4 *row = reinterpret_cast<const uint4 *>(&sm.xv[t][j * G]);
            const int rot = t + 2 * (j >> 1);
            __half2 mn2, mx2;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const uint4 w = row[(cc + rot) & 3];
                const __half2 v0 = bits_h2(w.x), v1 = bits_h2(w.y), v2 = bits_h2(w.z),
                              v3 = bits_h2(w.w);
                const __half2 lo = __hmin2(__hmin2(v0, v1), __hmin2(v2, v3));
                const __half2 hi = __hmax2(__hmax2(v0, v1), __hmax2(v2, v3));
                mn2 = cc == 0 ? lo : __hmin2(mn2, lo);
                mx2 = cc == 0 ? hi : __hmax2(mx2, hi);
            }
            mnb = __half_as_ushort(__hmin(__low2half(mn2), __high2half(mn2)));
            mxb = __half_as_ushort(__hmax(__low2half(mx2), __high2half(mx2)));
        }
        const GroupQ q = group_params<BITS>(h2fix(mnb), mnb, h2fix(mxb));
        if (i < D) {
            ksz[i] = q.scale_bits;
            ksz[D + i] = q.zero_bits;
        } else {
            const int a = i - D, t = a / NG, j = a % NG;
            vsz[j * G + t] = q.scale_bits;
            vsz[NG * G + j * G + t] = q.zero_bits;
        }
        sm.zfix[i] = q.zero_fix;
        sm.sfix[i] = q.scale_fix;
        sm.zf[i] = __half2float(__ushort_as_half(mnb));
        sm.sf[i] = __half2float(__ushort_as_half(q.scale_bits));
        // a zero scale gives a zero reciprocal, so the estimate below is 0 (code 0)
        sm.inv[i] = q.scale_fix ? 1.0f / __half2float(__ushort_as_half(q.scale_bits)) : 0.f;
    }
    __syncthreads();
    // 2. codes of the 2 * G * D elements, on packed fp32 pairs.  est =
    //    (x - zero) * (1 / scale) in fp32 is
    //    within 3e-6 of the true quotient while below cmax + 1 (three roundings of
    //    relative 2^-24 on a quotient of at most 16), so away from a rounding
    //    midpoint its nearest integer is the exact code.  Clamped to cmax, it is
    //    rounded half-even by adding 1.5 * 2^23 (the sum's low mantissa byte is the
    //    code); a word with an estimate within 1e-4 of a midpoint is redone in
    //    exact integer arithmetic (quant_code_inv).  A zero scale has a zero
    //    reciprocal: estimate 0, code 0.
    constexpr float MAGIC = 12582912.0f;   // 1.5 * 2^23: ulp 1 over [2^23, 2^24)
    constexpr float NEAR = 0.5f - 1e-4f;
    const float2 magic2 = make_float2(MAGIC, MAGIC);
    // est of a pair of elements, clamped; r holds the rounded codes, the return
    // value says whether either estimate lies near a midpoint
    auto pair_codes = [&](uint32_t x2, float2 z, float2 inv, float2 &r) -> bool {
        float2 e = fmul2(fsub2(__half22float2(bits_h2(x2)), z), inv);
        e = make_float2(fminf(e.x, (float)CMAX), fminf(e.y, (float)CMAX));
        r = fadd2(e, magic2);
        const float2 f = fsub2(e, fsub2(r, magic2));
        return fabsf(f.x) > NEAR || fabsf(f.y) > NEAR;
    };
    // 2a. 4-bit K token rows, straight into the block: field f of word w holds
    //     the code of channel 8w + f (one 16-byte chunk of inputs per word).
    //     2-bit words (16 channels) measured slower this way, and GEAR reads the
    //     K codes back as bytes; both are packed from bytes in 3a.
    constexpr int FPW = 32 / BITS;
    constexpr bool K_DIRECT = BITS == 4 && !GEAR;
    uint32_t *kw = reinterpret_cast<uint32_t *>(kblk);
    for (int i = threadIdx.x; K_DIRECT && i < G * WK; i += QTHREADS) {
        const int t = i / WK, c0 = FPW * (i % WK);
        uint32_t word = 0;
        bool near = false;
#pragma unroll
        for (int q = 0; q < FPW / 8; ++q) {
            const int c = c0 + 8 * q;
            const uint4 xw = *reinterpret_cast<const uint4 *>(&sm.xk[t][c]);
            const float4 za = *reinterpret_cast<const float4 *>(&sm.zf[c]);
            const float4 zb = *reinterpret_cast<const float4 *>(&sm.zf[c + 4]);
            const float4 ia = *reinterpret_cast<const float4 *>(&sm.inv[c]);
            const float4 ib = *reinterpret_cast<const float4 *>(&sm.inv[c + 4]);
            float2 r[4];
            near |= pair_codes(xw.x, make_float2(za.x, za.y), make_float2(ia.x, ia.y), r[0]);
            near |= pair_codes(xw.y, make_float2(za.z, za.w), make_float2(ia.z, ia.w), r[1]);
            near |= pair_codes(xw.z, make_float2(zb.x, zb.y), make_float2(ib.x, ib.y), r[2]);
            near |= pair_codes(xw.w, make_float2(zb.z, zb.w), make_float2(ib.z, ib.w), r[3]);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                word |= (__float_as_uint(r[u].x) & CMAX) << (BITS * (8 * q + 2 * u));
                word |= (__float_as_uint(r[u].y) & CMAX) << (BITS * (8 * q + 2 * u + 1));
            }
        }
        if (near) {
            word = 0;
            for (int f = 0; f < FPW; ++f)
                word |= (uint32_t)quant_code_inv(sm.xk[t][c0 + f], sm.zfix[c0 + f], sm.zf[c0 + f],
                                                 sm.sfix[c0 + f], sm.inv[c0 + f], CMAX)
                        << (BITS * f);
        }
        kw[i] = word;
    }
    // 2b. codes as bytes, four channels per step: the V elements (the four share
    //     one (token, channel group) set) and, unless 2a took them, the K elements
    for (int i = threadIdx.x; i < (K_DIRECT ? 1 : 2) * G * D / 4; i += QTHREADS) {
        const bool isk = !K_DIRECT && i >= G * D / 4;
        const int e = 4 * (isk ? i - G * D / 4 : i);
        const int t = e / D, d0 = e % D;
        const uint2 xw = *reinterpret_cast<const uint2 *>(isk ? &sm.xk[t][d0] : &sm.xv[t][d0]);
        float2 z01, z23, i01, i23;
        int pis[4];
        if (isk) {   // per-channel parameters of channels d0 .. d0 + 3
            const float4 z4 = *reinterpret_cast<const float4 *>(&sm.zf[d0]);
            const float4 i4 = *reinterpret_cast<const float4 *>(&sm.inv[d0]);
            z01 = make_float2(z4.x, z4.y), z23 = make_float2(z4.z, z4.w);
            i01 = make_float2(i4.x, i4.y), i23 = make_float2(i4.z, i4.w);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                pis[u] = d0 + u;
        } else {
            const int pi = D + t * NG + d0 / G;
            const float zz = sm.zf[pi], ii = sm.inv[pi];
            z01 = z23 = make_float2(zz, zz);
            i01 = i23 = make_float2(ii, ii);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                pis[u] = pi;
        }
        float2 r01, r23;
        const bool near = pair_codes(xw.x, z01, i01, r01) | pair_codes(xw.y, z23, i23, r23);
        uint32_t word = (__float_as_uint(r01.x) & 0xffu) | ((__float_as_uint(r01.y) & 0xffu) << 8) |
                        ((__float_as_uint(r23.x) & 0xffu) << 16) | (__float_as_uint(r23.y) << 24);
        if (near) {
            const uint16_t xs[4] = {(uint16_t)(xw.x & 0xffff), (uint16_t)(xw.x >> 16),
                                    (uint16_t)(xw.y & 0xffff), (uint16_t)(xw.y >> 16)};
            const float zs[4] = {z01.x, z01.y, z23.x, z23.y}, is[4] = {i01.x, i01.y, i23.x, i23.y};
            word = 0;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                word |= (uint32_t)quant_code_inv(xs[u], sm.zfix[pis[u]], zs[u], sm.sfix[pis[u]],
                                                 is[u], CMAX) << (8 * u);
        }
        *reinterpret_cast<uint32_t *>(isk ? &sm.ck[t][d0] : &sm.cv[t][d0]) = word;
    }
    __syncthreads();
    // 3a. K token rows from the bytes (2-bit, GEAR): field f of word w holds
    //     channel (32/BITS)*w + f
    for (int i = threadIdx.x; !K_DIRECT && i < G * WK; i += QTHREADS) {
        const int t = i / WK, w = i % WK;
        uint32_t word = 0;
#pragma unroll
        for (int f = 0; f < FPW; ++f)
            word |= (uint32_t)sm.ck[t][FPW * w + f] << (BITS * f);
        kw[i] = word;
    }
    // 3b. V token pairs: word ((rr + 2 pair) mod 8)*W + k, field j holds channel
    // 16*(k*(8/BITS) + j/2) + 8*(j%2) + rr; low half token 2i, high half 2i+1
    uint32_t *vw = reinterpret_cast<uint32_t *>(vblk);
    for (int i = threadIdx.x; i < (G / 2) * 8 * W; i += QTHREADS) {
        const int pair = i / (8 * W), rk = i % (8 * W), rr = rk / W, k = rk % W;
        const int slot = pair * 8 * W + ((rr + 2 * pair) & 7) * W + k;
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < 16 / BITS; ++j) {
            const int d = 16 * (k * (8 / BITS) + j / 2) + 8 * (j % 2) + rr;
            word |= (uint32_t)sm.cv[2 * pair][d] << (BITS * j);
            word |= (uint32_t)sm.cv[2 * pair + 1][d] << (16 + BITS * j);
        }
        vw[slot] = word;
    }
    __syncthreads();
    if (GEAR) {   // 4. the GEAR corrections of the group's quantisation residual
        gear_sides<D, BITS>(sm, *gs, kside, vside);
    }
}

// n_q (tokens quantised) at length T: 32 * floor(max(0, T - R) / 32).
__device__ __forceinline__ long kivi_nq(long T, int R)
{
    const long over = T - R;
    return over > 0 ? (over / KIVI_G) * KIVI_G : 0;
}

// Append n_new tokens to every unit of a KIVI cache.  GROUPS: CTA (unit, y)
// quantises the groups flushed by this append with index = y mod gridDim.y.
// RESIDUAL: the new tokens that stay fp16 are written to their ring slots.  A
// single launch may do both only when it is one CTA per unit (the ring slots
// it writes may be ones a flushed group still reads); bulk appends run the
// groups on a wide grid first and the residual in a second launch.
template <int D, int BITS, bool GROUPS, bool RESIDUAL, bool GEAR>
__global__ void __launch_bounds__(QTHREADS, GEAR ? 2 : 6)
    k_append_quant(int n_units, int Hkv, int R, int Cq, int n_new, const uint16_t *__restrict__ k_new,
                   const uint16_t *__restrict__ v_new, uint8_t *__restrict__ kb,
                   uint8_t *__restrict__ vb, uint16_t *__restrict__ k_res,
                   uint16_t *__restrict__ v_res, const int32_t *__restrict__ len,
                   const GroupBlocks blocks, uint8_t *__restrict__ kg, uint8_t *__restrict__ vg,
                   int *status)
{
    constexpr int G = KIVI_G;
    constexpr int NS = (2 * G * D + 99) / 100;
    constexpr long SIDE = (4 * NS + 4 * G + 4 * D + 15) / 16 * 16;
    __shared__ GroupSmem<D> sm;
    extern __shared__ __align__(16) uint8_t gear_dyn[];
    GearSmem<D> *gs = GEAR ? reinterpret_cast<GearSmem<D> *>(gear_dyn) : nullptr;

    // units blockIdx.x, blockIdx.x + gridDim.x, ... (decode-sized appends run one wave
    // of CTAs over all units; bulk appends one CTA column per unit)
    for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
    const int b = unit / Hkv;
    const int CR = R + G;
    const long T0 = len[b], T1 = T0 + n_new;
    const long nq0 = kivi_nq(T0, R), nq1 = kivi_nq(T1, R);
    if (nq1 > Cq) {
        if (threadIdx.x == 0 && blockIdx.y == 0 && (GROUPS || !RESIDUAL))
            flag_error(status, DEV_CAPACITY);
        continue;
    }
    const uint16_t *kn = k_new + (size_t)unit * n_new * D;
    const uint16_t *vn = v_new + (size_t)unit * n_new * D;

    if (GROUPS) {
        const uint16_t *kr = k_res + (size_t)unit * CR * D;
        const uint16_t *vr = v_res + (size_t)unit * CR * D;
        for (long g = nq0 / G + blockIdx.y; g < nq1 / G; g += gridDim.y) {
            const long long gi = blocks.index(unit, g);
            if (gi < 0) {   // no page behind this group: skip it, flag it
                if (threadIdx.x == 0)
                    flag_error(status, DEV_CAPACITY);
                continue;
            }
            const long long off = gi * blocks.block;
            pack_group<D, BITS, GEAR>(g, T0, CR, kn, vn, kr, vr, kb + off, vb + off, sm, gs,
                                      GEAR ? kg + gi * SIDE : nullptr,
                                      GEAR ? vg + gi * SIDE : nullptr);
        }
    }
    if (RESIDUAL) {
        // new tokens that stay in fp16 go to ring slot p mod (R + 32)
        const long r0 = nq1 > T0 ? nq1 : T0;
        uint4 *krw = reinterpret_cast<uint4 *>(k_res + (size_t)unit * CR * D);
        uint4 *vrw = reinterpret_cast<uint4 *>(v_res + (size_t)unit * CR * D);
        const long total = (T1 - r0) * (D / 8);
        for (long i = blockIdx.y * QTHREADS + threadIdx.x; i < total; i += gridDim.y * QTHREADS) {
            const long p = r0 + i / (D / 8);
            const int ch = (int)(i % (D / 8));
            const long slot = p % CR;
            krw[slot * (D / 8) + ch] = reinterpret_cast<const uint4 *>(kn + (p - T0) * D)[ch];
            vrw[slot * (D / 8) + ch] = reinterpret_cast<const uint4 *>(vn + (p - T0) * D)[ch];
        }
    }
    }   // units
}

__global__ void k_len_bump(int B, int n_new, int32_t *len)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < B)
        len[i] += n_new;
}

template <int D, int BITS, bool GEAR>
cudaError_t launch_quant_impl(const kvc_quant_cache &c, const uint16_t *k_new,
                              const uint16_t *v_new, int n_new, cudaStream_t s)
{
    const int units = c.B * c.Hkv;
    const GroupBlocks blocks{c.block_table, c.Cq / KIVI_G, c.num_pages,
                             KIVI_G * D * BITS / 8 + 4 * D};
    const int dyn = GEAR ? (int)sizeof(GearSmem<D>) : 0;
    if (GEAR) {   // the GEAR stage sits in dynamic shared memory next to the static group stage
        cudaError_t e = set_smem_once(
            reinterpret_cast<const void *>(k_append_quant<D, BITS, true, true, GEAR>), dyn);
        if (e == cudaSuccess)
            e = set_smem_once(
                reinterpret_cast<const void *>(k_append_quant<D, BITS, true, false, GEAR>), dyn);
        if (e != cudaSuccess)
            return e;
    }
    if (n_new <= KIVI_G) {
        // decode-sized: at most two groups flush per unit; one wave of CTAs walks the
        // units, each doing both parts for its units
        const int per_sm = GEAR ? 2 : 6;
        const int grid = units < per_sm * sm_count() ? units : per_sm * sm_count();
        k_append_quant<D, BITS, true, true, GEAR><<<grid, QTHREADS, dyn, s>>>(
            units, c.Hkv, c.R, c.Cq, n_new, k_new, v_new, c.k_blocks, c.v_blocks, c.k_res, c.v_res,
            c.len, blocks, c.k_gear, c.v_gear, dev_status_ptr());
    } else {
        // bulk: the flushed groups of every unit spread over the grid, then the residual
        const long max_groups = n_new / KIVI_G + 1;
        const long fill = (8L * sm_count() + units - 1) / units;  // >= ~8 CTAs per SM in total
        int gy = (int)(max_groups < fill ? max_groups : fill);
        gy = gy < 1 ? 1 : (gy > 65535 ? 65535 : gy);
        k_append_quant<D, BITS, true, false, GEAR><<<dim3(units, gy), QTHREADS, dyn, s>>>(
            units, c.Hkv, c.R, c.Cq, n_new, k_new, v_new, c.k_blocks, c.v_blocks, c.k_res, c.v_res,
            c.len, blocks, c.k_gear, c.v_gear, dev_status_ptr());
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
        k_append_quant<D, BITS, false, true, false><<<units, QTHREADS, 0, s>>>(
            units, c.Hkv, c.R, c.Cq, n_new, k_new, v_new, c.k_blocks, c.v_blocks, c.k_res, c.v_res,
            c.len, blocks, nullptr, nullptr, dev_status_ptr());
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    k_len_bump<<<(c.B + 255) / 256, 256, 0, s>>>(c.B, n_new, c.len);
    return cudaGetLastError();
}

template <int D, int BITS>
cudaError_t launch_quant_bits(const kvc_quant_cache &c, const uint16_t *k_new,
                              const uint16_t *v_new, int n_new, cudaStream_t s)
{
    return c.k_gear ? launch_quant_impl<D, BITS, true>(c, k_new, v_new, n_new, s)
                    : launch_quant_impl<D, BITS, false>(c, k_new, v_new, n_new, s);
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
            reinterpret_cast<uint4 *>(c.V), c.pos, c.n, c.seqlen,
            SlotRows{c.block_table, c.C, c.num_pages}, dev_status_ptr());
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
                                        SlotRows{c.block_table, c.C, c.num_pages},
                                        dev_status_ptr());
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    const int m = units > c.B ? units : c.B;
    k_append_bump<<<(m + 255) / 256, 256, 0, s>>>(c.B, c.Hkv, c.C, n_new, c.n, c.seqlen);
    return cudaGetLastError();
}

cudaError_t launch_stream_append(const kvc_slot_cache &c, const uint16_t *k_new,
                                 const uint16_t *v_new, int n_sink, int n_recent, cudaStream_t s)
{
    const int warps = c.Hkv < 16 ? c.Hkv : 16;
    k_stream_append<<<c.B, 32 * warps, 0, s>>>(
        c.Hkv, c.D, c.C, n_sink, n_recent, reinterpret_cast<const uint4 *>(k_new),
        reinterpret_cast<const uint4 *>(v_new), reinterpret_cast<uint4 *>(c.K),
        reinterpret_cast<uint4 *>(c.V), c.pos, c.n, c.seqlen,
        SlotRows{c.block_table, c.C, c.num_pages}, dev_status_ptr());
    return cudaGetLastError();
}

cudaError_t launch_append_quant(const kvc_quant_cache &c, const uint16_t *k_new,
                                const uint16_t *v_new, int n_new, cudaStream_t s)
{
    if (c.D == 128)
        return c.bits == 4 ? launch_quant_bits<128, 4>(c, k_new, v_new, n_new, s)
                           : launch_quant_bits<128, 2>(c, k_new, v_new, n_new, s);
    return c.bits == 4 ? launch_quant_bits<64, 4>(c, k_new, v_new, n_new, s)
                       : launch_quant_bits<64, 2>(c, k_new, v_new, n_new, s);
}

} // namespace kvc
