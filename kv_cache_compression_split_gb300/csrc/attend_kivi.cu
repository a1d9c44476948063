// attend_kivi.cu -- split-KV decode attention over a KIVI cache ("Rethinking KV
// Cache Compression" guide, §16 "4 种方法逐步执行": the decode read dequantises
// the old cache or uses a quantised kernel; the newest tokens stay in fp16).
//
// Work items are (sequence, KV head, split); persistent CTAs take them
// round-robin.  A producer lane streams the tiles of all its items into one
// shared-memory ring: quantised tiles of four 32-token groups (1-D bulk copies
// of the packed K and V group blocks) and, in the unit's last split, residual
// tiles of 32 fp16 ring slots (2-D TMA, 128-byte swizzle).  Four consumer
// warps work on a tile: warp w takes group w of a quantised tile, warps 0-1
// take 16 slots each of a residual tile.  Nothing is dequantised to memory:
//
//   K (per-channel scale s_d and zero z_d of the group):
//     q . k_t = sum_d (q_d s_d) c_{t,d} + sum_d q_d z_d
//   the scaled query q~ = q * s (binary16) is the B operand of S^T = C Q~^T
//   and the bias sum_d q_d z_d (fp32) is added to the scores.
//   V (per-token scale s_t and zero z_t of each 32-channel group):
//     sum_t p_t v_{t,d} = sum_t (p_t s_t) c_{t,d} + sum_t p_t z_t
//   p~ = p * s_t (binary16) is the B operand of O^T += C^T P~^T; the zero term
//   Z[group][head] = sum_t z_t p_t is one more MMA per 16 tokens.
//
// Codes enter the MMA as binary16 subnormals: masking a packed word leaves the
// bit pattern c << (bits*j), which reads as c * 2^(bits*j - 24) exactly, so a
// single AND per pair of codes is the whole conversion.  The power-of-two
// field weights are divided out of the K operand (q~ / 2^(bits*j)) or undone
// per output row at the end, and the 2^-24 is undone in the fp32 results.
//
// GEAR caches ("Rethinking KV Cache Compression" guide, §2: GEAR sparsity 2%,
// rank 2; §16: the corrections act on KIVI's quantisation residual) add, per
// group, x_hat = x_q + S + A^T B.  The same kernel handles them, again without
// dequantising: the quantised tile also carries the groups' side blocks, the
// sparse entries of a group are scattered into a per-warp fp16 tile (zero
// elsewhere) and the corrections are extra MMAs on fp32 accumulators:
//   scores  += S Q^T + A^T (B Q^T)        (B Q^T: 2 x heads)
//   O^T     += S^T P^T + B^T (A P^T)       (A P^T: 2 x heads)
// where the rank-2 products run as MMAs whose k dimension holds the two ranks.
#include "kvc_device.cuh"
#include "kvc_internal.h"

#include <math.h>

namespace kvc {

namespace {

constexpr int NCW = 4;
constexpr int NTHREADS = (NCW + 1) * 32;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
constexpr float TWO24 = 16777216.0f;
constexpr float TWOM24 = 1.0f / 16777216.0f;

template <int D, int BITS, bool GEAR = false> struct KiviCfg {
    static constexpr int G = KIVI_G;
    static constexpr int NG = D / G;                   // V channel groups
    static constexpr int WK = D * BITS / 32;           // words per K token row
    static constexpr int WPL = WK / 4;                 // K words per lane per row
    static constexpr int W = D * BITS / 128;           // V words per lane-row per pair
    static constexpr int FPW = 32 / BITS;              // fields per word
    static constexpr int HALF = FPW / 2;               // fields per 16-bit half
    static constexpr int MPW = 8 / BITS;               // V m-tiles per word
    static constexpr int CODE_BYTES = G * D * BITS / 8;
    static constexpr int BLOCK = CODE_BYTES + 4 * D;
    static constexpr int QG = NCW;                     // groups per quantised tile
    static_assert(QG == KIVI_PAGE_GROUPS, "a quantised tile is one page of the paged layout");
    static constexpr int NS = (2 * G * D + 99) / 100;  // GEAR sparse entries per group
    static constexpr int NSJ = (NS + 31) / 32;         // sparse entries per lane
    // GEAR side block: NS indices, NS values, A [2][G], B [2][D], padded to 16 bytes
    static constexpr int SIDE = GEAR ? (4 * NS + 4 * G + 4 * D + 15) / 16 * 16 : 0;
    static constexpr int SIDE_A = 4 * NS, SIDE_B = 4 * NS + 4 * G;   // byte offsets
    static_assert(SIDE_B == SIDE_A + 4 * G, "A [2][G] binary16 precedes B");
    static constexpr int QT_BYTES = 2 * QG * (BLOCK + SIDE);
    // ring slots per residual tile (16 for 2-bit codes, which would size the stages by the
    // smaller quantised tile and keep five in flight instead of three, measured 129 vs 119 us
    // on the 32-sequence MHA workload: the 2-bit read path is bound by instructions, not by
    // bytes in flight, and the extra residual tiles cost more than the deeper ring gains)
    static constexpr int RS = 32;
    static constexpr int NBOX = D / 64;
    static constexpr int RT_BYTES = 2 * RS * D * 2;
    static constexpr int STAGE_BYTES =
        ((QT_BYTES > RT_BYTES ? QT_BYTES : RT_BYTES) + 1023) / 1024 * 1024;
    // merge scratch: every warp's (m, l) per head, then per owner warp (OWN m-tiles of
    // output channels each) the other three warps' accumulators of those channels; rows
    // padded by 4 words (conflict-free fragment stores)
    static constexpr int OWN = (D / 16) / NCW;
    static constexpr int OSTR = 16 * OWN + 4;
    static constexpr int RED_BYTES = (NCW * 16 + NCW * (NCW - 1) * 8 * OSTR) * 4;
    // GEAR: one 32 x D fp16 sparse tile per consumer warp, rows padded by 16 bytes
    // (conflict-free ldmatrix)
    static constexpr int DT_STRIDE = (D + 8) * 2;
    static constexpr int DT_BYTES = GEAR ? NCW * G * DT_STRIDE : 0;
    // The plain query words of an item, one 16-byte chunk per (lane, 2 k-steps),
    // double-buffered (the next item's are written during the current one).  GEAR reads
    // them as the Q^T fragments of its correction MMAs; KIVI as the B operand of the
    // bias chain, when the buffers fit beside the stages it would have anyway (they
    // free 16 registers per thread that the 128-register cap of three CTAs per SM
    // would otherwise spill)
    // Where a second area fits too, KIVI also stages the scaled query pairs q / 2^(bits j)
    // of the K operand (16 more registers freed per thread).
    static constexpr int QCH = D / 32;                 // 16-byte chunks per lane
    static constexpr int QS_BUF = QCH * 32 * 16;       // one area: a chunk per (lane, k)
    // CTAs per SM: three for KIVI (each within a third of the SM's 228 KB of shared
    // memory, 1 KB of it reserved per CTA), two for GEAR
    static constexpr int CTAS = GEAR ? 2 : 3;
    static constexpr int KIVI_ROOM = 233472 / 3 - 1024 - RED_BYTES - 1024 - 64;
    static constexpr bool fits(int areas)
    {
        return (KIVI_ROOM - 2 * areas * QS_BUF) / STAGE_BYTES == KIVI_ROOM / STAGE_BYTES;
    }
    static constexpr int QS_AREAS = GEAR ? 1 : (fits(2) ? 2 : (fits(1) ? 1 : 0));
    static constexpr bool QS_BIAS = !GEAR && QS_AREAS >= 1;
    static constexpr bool QS_PAIRS = !GEAR && QS_AREAS == 2;
    static constexpr int QS_ITEM = QS_AREAS * QS_BUF;  // per item; two items in flight
    static constexpr int QS_BYTES = 2 * QS_ITEM;
    static constexpr int NSTAGE_PLAIN =
        GEAR ? ((81920 / STAGE_BYTES) < 3 ? 3 : (81920 / STAGE_BYTES))
             : (KIVI_ROOM - QS_BYTES) / STAGE_BYTES;
    // with the sparse tiles, as many stages as keep two CTAs resident per SM
    static constexpr int NSTAGE_FIT =
        (112640 - RED_BYTES - DT_BYTES - QS_BYTES - 1104) / STAGE_BYTES;
    static constexpr int NSTAGE =
        !GEAR ? NSTAGE_PLAIN
              : (NSTAGE_FIT < 2 ? 2 : (NSTAGE_FIT < NSTAGE_PLAIN ? NSTAGE_FIT : NSTAGE_PLAIN));
    static constexpr int SMEM =
        NSTAGE * STAGE_BYTES + RED_BYTES + DT_BYTES + QS_BYTES + 2 * NSTAGE * 8 + 1024;
};

struct KiviParams {
    int Hq, Hkv, g, Cq, R, CR;
    int splits, qtiles_per_split, n_items;
    int full_units;                 // units 0 .. full_units-1 run unsplit, the rest in `splits`
    const uint16_t *q;
    uint16_t *o;
    float *lse;
    const uint8_t *kb, *vb;
    const uint8_t *kg, *vg;         // GEAR side blocks, indexed like the group blocks
    GroupBlocks blocks;             // dense or paged group blocks
    const int32_t *len;
    float *part_o, *part_ml;
    float scale, scale_log2;
    int *status;
};

__device__ __forceinline__ void consumer_bar()
{
    asm volatile("bar.sync 1, %0;" ::"n"(NCW * 32) : "memory");
}

// Code field pair j (j < 16/BITS) of a packed word: fields j and j + 16/BITS
// (one per 16-bit half) masked in place.  Pairs j < 8/BITS come from w, the
// others from w >> 8, so a field never reaches the binary16 exponent: the bit
// pattern reads as two subnormals c_lo * 2^(BITS*(j mod 8/BITS) - 24), c_hi * (same).
template <int BITS> __device__ __forceinline__ uint32_t code_pair(uint32_t w, uint32_t w8, int j)
{
    constexpr int QUART = 8 / BITS;
    constexpr uint32_t M = ((1u << BITS) - 1) | (((1u << BITS) - 1) << 16);
    return (j < QUART ? w : w8) & (M << (BITS * (j % QUART)));
}

// Weight 2^(BITS * (j mod 8/BITS)) that code_pair leaves on field pair j (times 2^-24).
template <int BITS> __host__ __device__ constexpr float pair_weight(int j)
{
    return (float)(1u << (BITS * (j % (8 / BITS))));
}

// The K operand's query pairs of one lane: lane c covers channels [c D/4, (c+1) D/4)
// (w: those channels' words in order); pair pi holds channels (lo, lo + 16/BITS)
// divided by the pair's field weight 2^(BITS (pi mod 8/BITS)), in binary16.
template <int D, int BITS>
__device__ __forceinline__ void query_pairs(const uint32_t (&w)[D / 8], uint32_t (&qp)[D / 8])
{
    constexpr int FPW = 32 / BITS, HALF = FPW / 2;
#pragma unroll
    for (int pi = 0; pi < D / 8; ++pi) {
        const int j = pi % HALF;
        const int lo = FPW * (pi / HALF) + j, hi = lo + HALF;
        const __half2 wl = *reinterpret_cast<const __half2 *>(&w[lo >> 1]);
        const __half2 wh = *reinterpret_cast<const __half2 *>(&w[hi >> 1]);
        const float qlo = (lo & 1) ? __high2float(wl) : __low2float(wl);
        const float qhi = (hi & 1) ? __high2float(wh) : __low2float(wh);
        const float wgt = 1.0f / pair_weight<BITS>(j);
        qp[pi] = pack_half2(qlo * wgt, qhi * wgt);
    }
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b)
{
    __half2 r = __hmul2(*reinterpret_cast<const __half2 *>(&a), *reinterpret_cast<const __half2 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v)
{
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

__device__ __forceinline__ uint32_t pack_u16x2(uint16_t lo, uint16_t hi)
{
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

// Scatter the sparse entries of one GEAR side block into a warp's sparse tile:
// entry e (flat index t*D + d, binary16 value) lands at row t, column d.  The
// index is masked to the group, so a corrupt block cannot write outside the
// tile.  addr keeps the shared addresses for gear_clear.
template <int D, int NS, int NSJ, int STRIDE>
__device__ __forceinline__ void gear_scatter(const uint8_t *side, uint32_t tile, int lane,
                                             uint32_t (&addr)[NSJ])
{
    const uint16_t *idx = reinterpret_cast<const uint16_t *>(side);
    const uint16_t *val = idx + NS;
#pragma unroll
    for (int j = 0; j < NSJ; ++j) {
        const int e = lane + 32 * j;
        if (e < NS) {
            const uint32_t id = idx[e] & (KIVI_G * D - 1);
            addr[j] = tile + (id / D) * STRIDE + (id % D) * 2;
            st_shared_u16(addr[j], val[e]);
        }
    }
}

// Zero the entries gear_scatter wrote, leaving the tile all zero again.
template <int NS, int NSJ>
__device__ __forceinline__ void gear_clear(const uint32_t (&addr)[NSJ], int lane)
{
#pragma unroll
    for (int j = 0; j < NSJ; ++j)
        if (lane + 32 * j < NS)
            st_shared_u16(addr[j], 0);
}

// A rank x head product F held as an MMA result (row k = rank 0, 1 at lanes
// 4k + n/2, column n = head in register n % 2) turned into the B operand of an
// MMA whose k dimension is the rank: lane (n, 0) gets (F[0][n], F[1][n]), the
// other lanes zero (k >= 2).
__device__ __forceinline__ uint32_t rank2_b_operand(const float *f, int r, int c)
{
    const int src = r >> 1;
    const float x0 = __shfl_sync(0xffffffffu, f[0], src);
    const float x1 = __shfl_sync(0xffffffffu, f[1], src);
    const float y0 = __shfl_sync(0xffffffffu, f[0], 4 + src);
    const float y1 = __shfl_sync(0xffffffffu, f[1], 4 + src);
    return c == 0 ? pack_half2((r & 1) ? x1 : x0, (r & 1) ? y1 : y0) : 0u;
}

// N consecutive 32-bit words of shared memory (aligned to the widest of 16, 8 or
// 4 bytes that N allows) in as few loads as that alignment permits.
template <int N> __device__ __forceinline__ void lds_words(const uint32_t *src, uint32_t (&dst)[N])
{
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int e = 0; e < N / 4; ++e) {
            const uint4 v = reinterpret_cast<const uint4 *>(src)[e];
            dst[4 * e] = v.x;
            dst[4 * e + 1] = v.y;
            dst[4 * e + 2] = v.z;
            dst[4 * e + 3] = v.w;
        }
    } else if constexpr (N % 2 == 0) {
#pragma unroll
        for (int e = 0; e < N / 2; ++e) {
            const uint2 v = reinterpret_cast<const uint2 *>(src)[e];
            dst[2 * e] = v.x;
            dst[2 * e + 1] = v.y;
        }
    } else {
#pragma unroll
        for (int e = 0; e < N; ++e)
            dst[e] = src[e];
    }
}

struct KiviItem {
    int unit, split, nsplit, b, hk, T, n_groups, n_res, qt0, nq, nr;
};

// Work item -> (unit, split, splits of that unit).  Items 0 .. full_units-1 are
// whole units; the other units are split `splits` ways, and their items run
// split-major with the last split (the one that also holds the residual ring,
// so the largest) first: the CTAs that take items k, k + gridDim.x, ... then
// get a mix of splits whatever gridDim.x is, instead of all the last splits
// landing on the same CTAs.
__device__ __forceinline__ void kivi_unit_split(const KiviParams &p, int item, int &unit,
                                                int &split, int &nsplit)
{
    if (item < p.full_units) {
        unit = item;
        split = 0;
        nsplit = 1;
        return;
    }
    const int k = item - p.full_units;
    const int units = (p.n_items - p.full_units) / p.splits;
    const int s = k / units;
    unit = p.full_units + (k - s * units);
    split = p.splits - 1 - s;
    nsplit = p.splits;
}

template <int D, int BITS, bool GEAR>
__device__ __forceinline__ KiviItem kivi_item(const KiviParams &p, int item)
{
    using Cfg = KiviCfg<D, BITS, GEAR>;
    KiviItem w;
    kivi_unit_split(p, item, w.unit, w.split, w.nsplit);
    w.b = w.unit / p.Hkv;
    w.hk = w.unit % p.Hkv;
    w.T = p.len[w.b];
    const int over = w.T - p.R;
    w.n_groups = over > 0 ? over / Cfg::G : 0;
    if (w.n_groups * Cfg::G > p.Cq) {
        if (threadIdx.x == 0)
            flag_error(p.status, DEV_CAPACITY);
        w.n_groups = p.Cq / Cfg::G;
    }
    w.n_res = w.T - w.n_groups * Cfg::G;
    const int unit_qtiles = (w.n_groups + Cfg::QG - 1) / Cfg::QG;
    const int per = w.nsplit == 1 ? unit_qtiles : p.qtiles_per_split;
    w.qt0 = w.split * per;
    const int qt1 = min(unit_qtiles, w.qt0 + per);
    w.nq = qt1 > w.qt0 ? qt1 - w.qt0 : 0;
    w.nr = (w.split == w.nsplit - 1) ? (p.CR + Cfg::RS - 1) / Cfg::RS : 0;
    return w;
}

// Persistent CTAs: CTA k handles work items k, k + gridDim.x, ... (an item is one
// (sequence, KV head, split)); one TMA pipeline runs across all of its items.
template <int D, int BITS, bool GEAR>
__global__ void __launch_bounds__(NTHREADS, KiviCfg<D, BITS, GEAR>::CTAS)
    k_attend_kivi(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const KiviParams p)
{
    using Cfg = KiviCfg<D, BITS, GEAR>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_align1024(smem_raw);
    float *red = reinterpret_cast<float *>(smem + Cfg::NSTAGE * Cfg::STAGE_BYTES);
    uint8_t *dtiles = smem + Cfg::NSTAGE * Cfg::STAGE_BYTES + Cfg::RED_BYTES;
    uint8_t *qstage = dtiles + Cfg::DT_BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(qstage + Cfg::QS_BYTES);
    uint64_t *empty = full + Cfg::NSTAGE;
    __shared__ int s_abort;   // set when a wait ran out; every warp then stops
    volatile int *abort = &s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        s_abort = 0;
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
            prefetch_tmap(&tmV);
            int it = 0;
            for (int item = blockIdx.x; item < p.n_items; item += gridDim.x) {
                const KiviItem w = kivi_item<D, BITS, GEAR>(p, item);
                const int ntiles = w.nr + w.nq;   // residual tiles first, then quantised tiles
                for (int i = 0; i < ntiles; ++i, ++it) {
                    const int st = it % Cfg::NSTAGE;
                    if (it >= Cfg::NSTAGE &&
                        !mbar_wait_or_abort(&empty[st], ((it / Cfg::NSTAGE) & 1) ^ 1, abort)) {
                        flag_error(p.status, DEV_TIMEOUT);
                        return;
                    }
                    uint8_t *dst = smem + st * Cfg::STAGE_BYTES;
                    if (i < w.nr) {
                        mbar_arrive_expect_tx(&full[st], Cfg::RT_BYTES);
                        const int row = w.unit * p.CR + i * Cfg::RS;
#pragma unroll
                        for (int j = 0; j < Cfg::NBOX; ++j) {
                            tma_load_2d(dst + j * Cfg::RS * 128, &tmK, &full[st], 64 * j, row);
                            tma_load_2d(dst + (Cfg::NBOX + j) * Cfg::RS * 128, &tmV, &full[st],
                                        64 * j, row);
                        }
                    } else {
                        // a tile is 4 groups, one page in the paged layout
                        const int g0 = (w.qt0 + i - w.nr) * Cfg::QG;
                        const int ng = min(Cfg::QG, w.n_groups - g0);
                        const long long bi = p.blocks.index(w.unit, g0);
                        const long long off = bi * p.blocks.block;
                        if (bi < 0) {
                            // no page behind the tile: no copy, the stage completes empty
                            flag_error(p.status, DEV_CAPACITY);
                            mbar_arrive(&full[st]);
                        } else {
                            mbar_arrive_expect_tx(&full[st], 2 * ng * (Cfg::BLOCK + Cfg::SIDE));
                            bulk_load(dst, p.kb + off, ng * Cfg::BLOCK, &full[st]);
                            bulk_load(dst + Cfg::QG * Cfg::BLOCK, p.vb + off, ng * Cfg::BLOCK,
                                      &full[st]);
                            if constexpr (GEAR) {
                                // side blocks of the same groups, at the same pool index
                                const long long so = bi * Cfg::SIDE;
                                uint8_t *sd = dst + 2 * Cfg::QG * Cfg::BLOCK;
                                bulk_load(sd, p.kg + so, ng * Cfg::SIDE, &full[st]);
                                bulk_load(sd + Cfg::QG * Cfg::SIDE, p.vg + so, ng * Cfg::SIDE,
                                          &full[st]);
                            }
                        }
                    }
                }
            }
        }
        return;
    }

    const int r = lane >> 2, c = lane & 3, mi = lane >> 3, ri = lane & 7;
    const int h0 = 2 * c, h1 = 2 * c + 1;
    const bool hv = r < p.g;
    int it = 0;
    // GEAR: this warp's sparse tile, all zero between groups
    const uint32_t dt = smem_u32(dtiles) + warp * Cfg::G * Cfg::DT_STRIDE;
    // The query words of item `item` into q buffer qb, written by warp 0.  GEAR: the
    // Q^T B-operand fragments (head r: words 8s + c and 8s + c + 4 of the query row,
    // s = 0 .. D/16-1).  KIVI bias: the D/8 words of head r that lane c covers
    // (channels [c D/4, (c+1) D/4)) in order, chunk k holding the lane's words 4k .. 4k + 3.
    constexpr bool QSTAGE = GEAR || Cfg::QS_BIAS;
    auto stage_q = [&](int item, int qb) {
        int unit, split_unused, nsplit_unused;
        kivi_unit_split(p, item, unit, split_unused, nsplit_unused);
        const int bb = unit / p.Hkv, hh = unit % p.Hkv;
        const uint32_t *q32 = reinterpret_cast<const uint32_t *>(
            p.q + ((size_t)bb * p.Hq + hh * p.g + (hv ? r : 0)) * D);
        uint4 *dst = reinterpret_cast<uint4 *>(qstage + qb * Cfg::QS_ITEM) + lane;
        if constexpr (GEAR) {
#pragma unroll
            for (int k = 0; k < Cfg::QCH; ++k)
                dst[32 * k] = hv ? make_uint4(q32[16 * k + c], q32[16 * k + c + 4],
                                              q32[16 * k + 8 + c], q32[16 * k + 12 + c])
                                 : make_uint4(0u, 0u, 0u, 0u);
        } else {
            uint32_t w[D / 8];
#pragma unroll
            for (int e = 0; e < D / 8; ++e)
                w[e] = hv ? q32[c * (D / 8) + e] : 0u;
#pragma unroll
            for (int k = 0; k < Cfg::QCH; ++k)
                dst[32 * k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
            if constexpr (Cfg::QS_PAIRS) {
                uint32_t qp[D / 8];
                query_pairs<D, BITS>(w, qp);
#pragma unroll
                for (int k = 0; k < Cfg::QCH; ++k)
                    dst[32 * (Cfg::QCH + k)] =
                        make_uint4(qp[4 * k], qp[4 * k + 1], qp[4 * k + 2], qp[4 * k + 3]);
            }
        }
    };
    if constexpr (GEAR) {
        uint4 *z = reinterpret_cast<uint4 *>(dtiles + warp * Cfg::G * Cfg::DT_STRIDE);
        for (int e = lane; e < Cfg::G * Cfg::DT_STRIDE / 16; e += 32)
            z[e] = make_uint4(0u, 0u, 0u, 0u);
        __syncwarp();
    }
    if constexpr (QSTAGE) {
        if (warp == 0 && (int)blockIdx.x < p.n_items)
            stage_q(blockIdx.x, 0);
        consumer_bar();
    }
    int qbuf = 0;   // q buffer of the current item

    for (int item = blockIdx.x; item < p.n_items; item += gridDim.x, qbuf ^= 1) {
    const KiviItem wi = kivi_item<D, BITS, GEAR>(p, item);
    const int b = wi.b, hk = wi.hk, T = wi.T, n_groups = wi.n_groups, n_res = wi.n_res;
    const int qt0 = wi.qt0, nr = wi.nr, ntiles = wi.nr + wi.nq;
    const uint16_t *qrow = p.q + ((size_t)b * p.Hq + hk * p.g + (hv ? r : 0)) * D;
    float acc[D / 16][4];
#pragma unroll
    for (int m = 0; m < D / 16; ++m)
        acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.f;
    float zacc[2] = {0.f, 0.f};   // Z[group r][heads 2c, 2c+1] (meaningful for r < NG)
    float m_run0 = -INFINITY, m_run1 = -INFINITY, l_run0 = 0.f, l_run1 = 0.f;

    // online-softmax update over the scores a lane holds (N values per head);
    // x*: log2-domain scores of heads 2c (xa) and 2c+1 (xb); p* returns exp2(x - m)
    auto softmax_update = [&](auto &xa, auto &xb, int N) {
        float mx0 = xa[0], mx1 = xb[0];
#pragma unroll
        for (int e = 1; e < 4; ++e)
            if (e < N) {
                mx0 = fmaxf(mx0, xa[e]);
                mx1 = fmaxf(mx1, xb[e]);
            }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m_run0, mx0), mn1 = fmaxf(m_run1, mx1);
        const bool z0 = mn0 == -INFINITY, z1 = mn1 == -INFINITY;
        const float al0 = z0 ? 1.f : ex2(m_run0 - mn0);
        const float al1 = z1 ? 1.f : ex2(m_run1 - mn1);
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e)
            if (e < N) {
                xa[e] = z0 ? 0.f : ex2(xa[e] - mn0);
                xb[e] = z1 ? 0.f : ex2(xb[e] - mn1);
                s0 += xa[e];
                s1 += xb[e];
            }
        m_run0 = mn0;
        m_run1 = mn1;
        l_run0 = l_run0 * al0 + s0;
        l_run1 = l_run1 * al1 + s1;
        if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
            for (int m = 0; m < D / 16; ++m) {
                acc[m][0] *= al0;
                acc[m][1] *= al1;
                acc[m][2] *= al0;
                acc[m][3] *= al1;
            }
            zacc[0] *= al0;
            zacc[1] *= al1;
        }
    };

    int i = 0;
    // ======================= fp16 residual tiles (last split only)
    if (nr > 0) {
        // Q^T as the B operand: Q[head r][16s + 2c, +1] and [16s + 2c + 8, +1]
        uint32_t qf[D / 16][2];
        {
            const uint32_t *q32 = reinterpret_cast<const uint32_t *>(qrow);
#pragma unroll
            for (int s = 0; s < D / 16; ++s) {
                qf[s][0] = hv ? q32[8 * s + c] : 0u;
                qf[s][1] = hv ? q32[8 * s + c + 4] : 0u;
            }
        }
        for (; i < nr; ++i, ++it) {
            const int st = it % Cfg::NSTAGE;
            if (!mbar_wait_or_abort(&full[st], (it / Cfg::NSTAGE) & 1, abort)) {
                flag_error(p.status, DEV_TIMEOUT);
                i = ntiles + 1;
                break;
            }
            // RS/16 warps take 16 ring slots each; the warp groups take the tiles in turn
            constexpr int PW = Cfg::RS / 16, NPG = NCW / PW;
            static_assert(NCW % PW == 0, "whole warp groups per residual tile");
            const int wl = warp % PW;
            const int s0 = i * Cfg::RS + 16 * wl;
            if (warp / PW == i % NPG && s0 < p.CR) {
                const uint32_t kbase = smem_u32(smem + st * Cfg::STAGE_BYTES);
                const uint32_t vbase = kbase + Cfg::NBOX * Cfg::RS * 128;
                float sa[4] = {0.f, 0.f, 0.f, 0.f};
                const int krow = 16 * wl + ri + 8 * (mi & 1);
#pragma unroll
                for (int s = 0; s < D / 16; ++s) {
                    const int ch = 2 * s + (mi >> 1);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(swz128(kbase + (ch >> 3) * Cfg::RS * 128, krow, ch & 7), a0, a1, a2, a3);
                    mma16816(sa, a0, a1, a2, a3, qf[s][0], qf[s][1]);
                }
                const int ta = s0 + r, tb = s0 + r + 8;
                const bool va = ta < p.CR && ((T - 1 - ta) % p.CR + p.CR) % p.CR < n_res;
                const bool vb = tb < p.CR && ((T - 1 - tb) % p.CR + p.CR) % p.CR < n_res;
                float xa[2] = {va ? sa[0] * p.scale_log2 : -INFINITY, vb ? sa[2] * p.scale_log2 : -INFINITY};
                float xb[2] = {va ? sa[1] * p.scale_log2 : -INFINITY, vb ? sa[3] * p.scale_log2 : -INFINITY};
                softmax_update(xa, xb, 2);
                const uint32_t pb0 = movmatrix_t(pack_half2(xa[0], xb[0]));
                const uint32_t pb1 = movmatrix_t(pack_half2(xa[1], xb[1]));
                const int vrow = 16 * wl + ri + 8 * (mi >> 1);
#pragma unroll
                for (int m = 0; m < D / 16; ++m) {
                    const int ch = 2 * m + (mi & 1);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_t(swz128(vbase + (ch >> 3) * Cfg::RS * 128, vrow, ch & 7), a0, a1, a2, a3);
                    mma16816(acc[m], a0, a1, a2, a3, pb0, pb1);
                }
            }
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[st]);
        }
    }

    // ======================= quantised tiles: warp w takes group w (32 tokens)
    // query pairs: lane c covers channels [c D/4, (c+1) D/4); pair pi holds channels
    // (lo, lo + HALF) divided by the pair's field weight
    // (staged: read per group from shared memory instead)
    uint32_t qpair[Cfg::QS_PAIRS ? 1 : D / 8];
    // KIVI without the staged query: the same channels in order (for the bias)
    uint32_t qh[QSTAGE ? 1 : D / 8];
    if constexpr (!Cfg::QS_PAIRS) {
        uint32_t qh_[D / 8];
        const uint32_t *q32 = reinterpret_cast<const uint32_t *>(qrow + c * (D / 4));
#pragma unroll
        for (int e = 0; e < D / 8; ++e) {
            qh_[e] = hv ? q32[e] : 0u;
            if constexpr (!QSTAGE)
                qh[e] = qh_[e];
        }
        query_pairs<D, BITS>(qh_, qpair);
    }
    bool code_units = false;   // acc scaled to the quantised tiles' units
    for (; i < ntiles; ++i, ++it) {
        const int st = it % Cfg::NSTAGE;
        if (!mbar_wait_or_abort(&full[st], (it / Cfg::NSTAGE) & 1, abort)) {
            flag_error(p.status, DEV_TIMEOUT);
            break;
        }
        const int g0 = (qt0 + i - nr) * Cfg::QG;
        if (g0 + warp < n_groups) {
            if (!code_units) {
#pragma unroll
                for (int m = 0; m < D / 16; ++m) {
                    const int jj = m % Cfg::MPW;
                    const float wr = pair_weight<BITS>(2 * jj) * TWOM24;
                    const float wr8 = pair_weight<BITS>(2 * jj + 1) * TWOM24;
                    acc[m][0] *= wr;
                    acc[m][1] *= wr;
                    acc[m][2] *= wr8;
                    acc[m][3] *= wr8;
                }
                code_units = true;
            }
            const uint8_t *tile = smem + st * Cfg::STAGE_BYTES;
            const uint8_t *kblk = tile + warp * Cfg::BLOCK;
            const uint8_t *vblk = tile + (Cfg::QG + warp) * Cfg::BLOCK;
            const uint32_t *ksz = reinterpret_cast<const uint32_t *>(kblk + Cfg::CODE_BYTES);
            const uint32_t *vss = reinterpret_cast<const uint32_t *>(vblk + Cfg::CODE_BYTES);
            const uint32_t *vzz = vss + Cfg::NG * Cfg::G / 2;
            // GEAR side blocks of this warp's group; the K entries go into the tile now
            const uint8_t *kside = tile + 2 * Cfg::QG * Cfg::BLOCK + warp * Cfg::SIDE;
            const uint8_t *vside = kside + Cfg::QG * Cfg::SIDE;
            uint32_t saddr[Cfg::NSJ];
            if constexpr (GEAR)
                gear_scatter<D, Cfg::NS, Cfg::NSJ, Cfg::DT_STRIDE>(kside, dt, lane, saddr);

            // ---- the bias beta_h = sum_d q_hd z_d of the K zeros.  GEAR: one MMA chain over
            // the plain query Q^T whose A rows 0, 1 hold B (U = B Q^T) and row 2 the zeros,
            // with the sparse tile's S Q^T alongside.  KIVI: an MMA chain whose A rows 0-7
            // all hold the zeros, so every result row is beta; the k order is permuted so
            // that lane c's channels are the 32 it already holds (words 16c .. 16c + 15
            // of both rows, k-step s taking words 2s and 2s + 1).
            float dk0[4] = {0.f, 0.f, 0.f, 0.f}, dk1[4] = {0.f, 0.f, 0.f, 0.f};
            float uf[4] = {0.f, 0.f, 0.f, 0.f};   // rows 0-2: U, beta (GEAR)
            float ug[4] = {0.f, 0.f, 0.f, 0.f};   // (odd k-steps: a second chain)
            float bias0, bias1;   // log2-domain bias of heads 2c, 2c+1
            if constexpr (GEAR) {
                __syncwarp();   // every lane's K entries are in the tile
                uint4 qv[Cfg::QCH];
                const uint4 *qsrc =
                    reinterpret_cast<const uint4 *>(qstage + qbuf * Cfg::QS_ITEM) + lane;
#pragma unroll
                for (int k = 0; k < Cfg::QCH; ++k)
                    qv[k] = qsrc[32 * k];
                const uint32_t *arow =
                    r == 2 ? ksz + D / 2
                           : reinterpret_cast<const uint32_t *>(kside + Cfg::SIDE_B) + r * (D / 2);
                const bool ra = r <= 2;
#pragma unroll
                for (int s = 0; s < D / 16; ++s) {
                    // Q^T as the B operand: Q[head r][16s + 2c, +1] and [16s + 2c + 8, +1]
                    const uint32_t q0 = (s & 1) ? qv[s >> 1].z : qv[s >> 1].x;
                    const uint32_t q1 = (s & 1) ? qv[s >> 1].w : qv[s >> 1].y;
                    mma16816((s & 1) ? ug : uf, ra ? arow[8 * s + c] : 0u, 0u,
                             ra ? arow[8 * s + 4 + c] : 0u, 0u, q0, q1);
                    const int ch = 2 * s + (mi >> 1);
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(dt + (ri + 8 * (mi & 1)) * Cfg::DT_STRIDE + ch * 16, a0, a1, a2, a3);
                    mma16816(dk0, a0, a1, a2, a3, q0, q1);
                    ldsm_x4(dt + (16 + ri + 8 * (mi & 1)) * Cfg::DT_STRIDE + ch * 16, a0, a1, a2,
                            a3);
                    mma16816(dk1, a0, a1, a2, a3, q0, q1);
                }
                uf[0] += ug[0];
                uf[1] += ug[1];
                // beta of heads 2c, 2c+1: row 2 of the result, lane 8 + c
                bias0 = __shfl_sync(0xffffffffu, uf[0], 8 + c) * p.scale_log2;
                bias1 = __shfl_sync(0xffffffffu, uf[1], 8 + c) * p.scale_log2;
            } else {
                const uint4 *zl = reinterpret_cast<const uint4 *>(ksz + D / 2 + c * (D / 8));
                const uint4 *qsrc =
                    reinterpret_cast<const uint4 *>(qstage + qbuf * Cfg::QS_ITEM) + lane;
                float bz0[4] = {0.f, 0.f, 0.f, 0.f}, bz1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int e = 0; e < D / 32; ++e) {
                    const uint4 z4 = zl[e];
                    uint4 q4;
                    if constexpr (QSTAGE)
                        q4 = qsrc[32 * e];
                    else
                        q4 = make_uint4(qh[4 * e], qh[4 * e + 1], qh[4 * e + 2], qh[4 * e + 3]);
                    mma16816(bz0, z4.x, 0u, z4.y, 0u, q4.x, q4.y);
                    mma16816(bz1, z4.z, 0u, z4.w, 0u, q4.z, q4.w);
                }
                bias0 = (bz0[0] + bz1[0]) * p.scale_log2;
                bias1 = (bz0[1] + bz1[1]) * p.scale_log2;
            }
            // ---- q~ pairs (B operand)
            uint32_t qt[D / 8];
            {
                uint32_t qps[Cfg::QS_PAIRS ? D / 8 : 1];
                if constexpr (Cfg::QS_PAIRS) {
                    const uint4 *qsp = reinterpret_cast<const uint4 *>(
                                           qstage + qbuf * Cfg::QS_ITEM + Cfg::QS_BUF) + lane;
#pragma unroll
                    for (int k = 0; k < Cfg::QCH; ++k) {
                        const uint4 v = qsp[32 * k];
                        qps[4 * k] = v.x;
                        qps[4 * k + 1] = v.y;
                        qps[4 * k + 2] = v.z;
                        qps[4 * k + 3] = v.w;
                    }
                }
                const uint32_t *qsrc_pairs = Cfg::QS_PAIRS ? qps : qpair;
                const uint4 *sl = reinterpret_cast<const uint4 *>(ksz + c * (D / 8));
                uint32_t sw[D / 8];
#pragma unroll
                for (int e = 0; e < D / 32; ++e) {
                    const uint4 s4 = sl[e];
                    sw[4 * e] = s4.x;
                    sw[4 * e + 1] = s4.y;
                    sw[4 * e + 2] = s4.z;
                    sw[4 * e + 3] = s4.w;
                }
#pragma unroll
                for (int pi = 0; pi < D / 8; ++pi) {
                    const int lo = Cfg::FPW * (pi / Cfg::HALF) + pi % Cfg::HALF;
                    const int hi = lo + Cfg::HALF;
                    const uint32_t sp = __byte_perm(sw[lo >> 1], sw[hi >> 1],
                                                    ((lo & 1) ? 0x0032 : 0x0010) |
                                                        ((hi & 1) ? 0x7600 : 0x5400));
                    qt[pi] = hmul2_u32(qsrc_pairs[pi], sp);
                }
            }
            const float sk = TWO24 * p.scale_log2;

            // ---- S^T = C_K Q~^T for both 16-token row blocks of the group
            float sa0[4] = {0.f, 0.f, 0.f, 0.f}, sa1[4] = {0.f, 0.f, 0.f, 0.f};
            {
                const uint32_t *kw = reinterpret_cast<const uint32_t *>(kblk);
                uint32_t w0[Cfg::WPL], w1[Cfg::WPL], w2[Cfg::WPL], w3[Cfg::WPL];
                lds_words(kw + r * Cfg::WK + c * Cfg::WPL, w0);
                lds_words(kw + (r + 8) * Cfg::WK + c * Cfg::WPL, w1);
                lds_words(kw + (r + 16) * Cfg::WK + c * Cfg::WPL, w2);
                lds_words(kw + (r + 24) * Cfg::WK + c * Cfg::WPL, w3);
#pragma unroll
                for (int s = 0; s < D / 16; ++s) {
                    const int pa = 2 * s, pb = 2 * s + 1;
                    const int ka = pa / Cfg::HALF, kb2 = pb / Cfg::HALF;
                    const int ja = pa % Cfg::HALF, jb = pb % Cfg::HALF;
                    mma16816(sa0, code_pair<BITS>(w0[ka], w0[ka] >> 8, ja),
                             code_pair<BITS>(w1[ka], w1[ka] >> 8, ja),
                             code_pair<BITS>(w0[kb2], w0[kb2] >> 8, jb),
                             code_pair<BITS>(w1[kb2], w1[kb2] >> 8, jb), qt[pa], qt[pb]);
                    mma16816(sa1, code_pair<BITS>(w2[ka], w2[ka] >> 8, ja),
                             code_pair<BITS>(w3[ka], w3[ka] >> 8, ja),
                             code_pair<BITS>(w2[kb2], w2[kb2] >> 8, jb),
                             code_pair<BITS>(w3[kb2], w3[kb2] >> 8, jb), qt[pa], qt[pb]);
                }
            }
            // scores of heads 2c (xa) and 2c+1 (xb) at tokens r, r+8, 16+r, 24+r
            float xa[4] = {fmaf(sa0[0], sk, bias0), fmaf(sa0[2], sk, bias0),
                           fmaf(sa1[0], sk, bias0), fmaf(sa1[2], sk, bias0)};
            float xb[4] = {fmaf(sa0[1], sk, bias1), fmaf(sa0[3], sk, bias1),
                           fmaf(sa1[1], sk, bias1), fmaf(sa1[3], sk, bias1)};
            if constexpr (GEAR) {
                // ---- GEAR score correction  S Q^T + A^T U  (fp32, plain units)
                const uint32_t ub = rank2_b_operand(uf, r, c);
                const uint16_t *ak = reinterpret_cast<const uint16_t *>(kside + Cfg::SIDE_A);
                const bool c0 = c == 0;
                mma16816(dk0, c0 ? pack_u16x2(ak[r], ak[Cfg::G + r]) : 0u,
                         c0 ? pack_u16x2(ak[r + 8], ak[Cfg::G + r + 8]) : 0u, 0u, 0u, ub, 0u);
                mma16816(dk1, c0 ? pack_u16x2(ak[r + 16], ak[Cfg::G + r + 16]) : 0u,
                         c0 ? pack_u16x2(ak[r + 24], ak[Cfg::G + r + 24]) : 0u, 0u, 0u, ub, 0u);
                const float sl = p.scale_log2;
                xa[0] = fmaf(dk0[0], sl, xa[0]);
                xa[1] = fmaf(dk0[2], sl, xa[1]);
                xa[2] = fmaf(dk1[0], sl, xa[2]);
                xa[3] = fmaf(dk1[2], sl, xa[3]);
                xb[0] = fmaf(dk0[1], sl, xb[0]);
                xb[1] = fmaf(dk0[3], sl, xb[1]);
                xb[2] = fmaf(dk1[1], sl, xb[2]);
                xb[3] = fmaf(dk1[3], sl, xb[3]);
                // swap the K entries for the V entries
                __syncwarp();
                gear_clear<Cfg::NS, Cfg::NSJ>(saddr, lane);
                __syncwarp();
                gear_scatter<D, Cfg::NS, Cfg::NSJ, Cfg::DT_STRIDE>(vside, dt, lane, saddr);
            }
            softmax_update(xa, xb, 4);

            const uint32_t *vw = reinterpret_cast<const uint32_t *>(vblk);
            uint32_t pbs[2][2];   // P^T fragments of both 16-token blocks (GEAR)
#pragma unroll
            for (int rb = 0; rb < 2; ++rb) {
                // P^T fragments: pb0 = p[tokens 2c, 2c+1][head r], pb1 = tokens 2c+8, 2c+9
                const uint32_t pb0 = movmatrix_t(pack_half2(xa[2 * rb], xb[2 * rb]));
                const uint32_t pb1 = movmatrix_t(pack_half2(xa[2 * rb + 1], xb[2 * rb + 1]));
                pbs[rb][0] = pb0;
                pbs[rb][1] = pb1;
                const int t0 = 16 * rb + 2 * c;
                // zero term Z[group][head] += sum_t z_t p_t (A rows = channel groups)
                {
                    const bool zr = r < Cfg::NG;
                    const uint32_t za0 = zr ? vzz[(r * Cfg::G + t0) >> 1] : 0u;
                    const uint32_t za2 = zr ? vzz[(r * Cfg::G + t0 + 8) >> 1] : 0u;
                    float zc[4] = {zacc[0], zacc[1], 0.f, 0.f};
                    mma16816(zc, za0, 0u, za2, 0u, pb0, pb1);
                    zacc[0] = zc[0];
                    zacc[1] = zc[1];
                }
                // p~ = p * s_V per channel group (B operands)
                uint32_t ptb0[Cfg::NG], ptb1[Cfg::NG];
#pragma unroll
                for (int gd = 0; gd < Cfg::NG; ++gd) {
                    ptb0[gd] = hmul2_u32(pb0, vss[(gd * Cfg::G + t0) >> 1]);
                    ptb1[gd] = hmul2_u32(pb1, vss[(gd * Cfg::G + t0 + 8) >> 1]);
                }
                // O^T += C_V^T P~^T, m-tile m in channel group m/2; pair chunks are
                // stored rotated by twice the pair index
                const int pc = 8 * rb + c, pd = pc + 4;
                uint32_t wa[Cfg::W], wb[Cfg::W];
                lds_words(vw + pc * 2 * Cfg::WK + ((r + 2 * pc) & 7) * Cfg::W, wa);
                lds_words(vw + pd * 2 * Cfg::WK + ((r + 2 * pd) & 7) * Cfg::W, wb);
#pragma unroll
                for (int m = 0; m < D / 16; ++m) {
                    const int k = m / Cfg::MPW, jj = m % Cfg::MPW;
                    mma16816(acc[m], code_pair<BITS>(wa[k], wa[k] >> 8, 2 * jj),
                             code_pair<BITS>(wa[k], wa[k] >> 8, 2 * jj + 1),
                             code_pair<BITS>(wb[k], wb[k] >> 8, 2 * jj),
                             code_pair<BITS>(wb[k], wb[k] >> 8, 2 * jj + 1), ptb0[m / 2],
                             ptb1[m / 2]);
                }
            }
            if constexpr (GEAR) {
                // ---- GEAR output correction  S^T P^T + B^T (A P^T), added in code units
                __syncwarp();   // every lane's V entries are in the tile
                const bool rk = r < 2, c0 = c == 0;
                const uint32_t *av = reinterpret_cast<const uint32_t *>(vside + Cfg::SIDE_A);
                float wf[4] = {0.f, 0.f, 0.f, 0.f};   // W = A P^T: rank rows 0, 1
#pragma unroll
                for (int rb = 0; rb < 2; ++rb)
                    mma16816(wf, rk ? av[r * (Cfg::G / 2) + 8 * rb + c] : 0u, 0u,
                             rk ? av[r * (Cfg::G / 2) + 8 * rb + 4 + c] : 0u, 0u, pbs[rb][0],
                             pbs[rb][1]);
                const uint32_t wbo = rank2_b_operand(wf, r, c);
                const uint16_t *bv = reinterpret_cast<const uint16_t *>(vside + Cfg::SIDE_B);
#pragma unroll
                for (int m = 0; m < D / 16; ++m) {
                    float t4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int rb = 0; rb < 2; ++rb) {
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4_t(dt + (16 * rb + ri + 8 * (mi >> 1)) * Cfg::DT_STRIDE +
                                      (2 * m + (mi & 1)) * 16,
                                  a0, a1, a2, a3);
                        mma16816(t4, a0, a1, a2, a3, pbs[rb][0], pbs[rb][1]);
                    }
                    const int d = 16 * m + r;
                    mma16816(t4, c0 ? pack_u16x2(bv[d], bv[D + d]) : 0u,
                             c0 ? pack_u16x2(bv[d + 8], bv[D + d + 8]) : 0u, 0u, 0u, wbo, 0u);
                    const int jj = m % Cfg::MPW;
                    const float wr = pair_weight<BITS>(2 * jj) * TWOM24;
                    const float wr8 = pair_weight<BITS>(2 * jj + 1) * TWOM24;
                    acc[m][0] = fmaf(t4[0], wr, acc[m][0]);
                    acc[m][1] = fmaf(t4[1], wr, acc[m][1]);
                    acc[m][2] = fmaf(t4[2], wr8, acc[m][2]);
                    acc[m][3] = fmaf(t4[3], wr8, acc[m][3]);
                }
                __syncwarp();
                gear_clear<Cfg::NS, Cfg::NSJ>(saddr, lane);
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[st]);
    }

    // ---------------- back to plain units, add the zero term, merge the warps
    if (code_units) {
#pragma unroll
        for (int m = 0; m < D / 16; ++m) {
            const int jj = m % Cfg::MPW;
            const float wr = TWO24 / pair_weight<BITS>(2 * jj);
            const float wr8 = TWO24 / pair_weight<BITS>(2 * jj + 1);
            acc[m][0] *= wr;
            acc[m][1] *= wr;
            acc[m][2] *= wr8;
            acc[m][3] *= wr8;
        }
    }
#pragma unroll
    for (int gd = 0; gd < Cfg::NG; ++gd) {
        const float z0 = __shfl_sync(0xffffffffu, zacc[0], 4 * gd + c);
        const float z1 = __shfl_sync(0xffffffffu, zacc[1], 4 * gd + c);
#pragma unroll
        for (int mm = 0; mm < 2; ++mm) {
            acc[2 * gd + mm][0] += z0;
            acc[2 * gd + mm][1] += z1;
            acc[2 * gd + mm][2] += z0;
            acc[2 * gd + mm][3] += z1;
        }
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l_run0 += __shfl_xor_sync(0xffffffffu, l_run0, off);
        l_run1 += __shfl_xor_sync(0xffffffffu, l_run1, off);
    }
    if constexpr (QSTAGE) {
        // the next item's query words go to the other buffer: its readers finished
        // before the previous merge, and this item's readers before the barrier below
        if (warp == 0 && item + (int)gridDim.x < p.n_items)
            stage_q(item + gridDim.x, qbuf ^ 1);
    }
    consumer_bar();   // every warp has finished reading the previous item's scratch
    if (*abort)
        break;        // every consumer warp sees the same flag after the barrier
    // Each warp merges the output channels of its own m-tiles: it publishes its (m, l)
    // and hands the accumulators of the other warps' m-tiles to their owners.
    constexpr int MT = D / 16, OWN = Cfg::OWN, OSTR = Cfg::OSTR;
    float *const mlb = red;                 // [NCW][8 heads][m, l]
    float *const ob = red + NCW * 16;       // [owner][source slot][8 heads][OSTR]
    if (r == 0) {
        mlb[(warp * 8 + h0) * 2] = m_run0;
        mlb[(warp * 8 + h0) * 2 + 1] = l_run0;
        mlb[(warp * 8 + h1) * 2] = m_run1;
        mlb[(warp * 8 + h1) * 2 + 1] = l_run1;
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const int ow = m / OWN;
        if (ow == warp)
            continue;
        const int slot = warp < ow ? warp : warp - 1;
        float *dst = ob + (ow * (NCW - 1) + slot) * 8 * OSTR + (m - ow * OWN) * 16;
        dst[h0 * OSTR + r] = acc[m][0];
        dst[h1 * OSTR + r] = acc[m][1];
        dst[h0 * OSTR + r + 8] = acc[m][2];
        dst[h1 * OSTR + r + 8] = acc[m][3];
    }
    consumer_bar();
    {
        // the warps' weights, summed in warp order
        float ms0 = mlb[h0 * 2], ms1 = mlb[h1 * 2];
#pragma unroll
        for (int v = 1; v < NCW; ++v) {
            ms0 = fmaxf(ms0, mlb[(v * 8 + h0) * 2]);
            ms1 = fmaxf(ms1, mlb[(v * 8 + h1) * 2]);
        }
        float sc0[NCW], sc1[NCW], ls0 = 0.f, ls1 = 0.f;
#pragma unroll
        for (int v = 0; v < NCW; ++v) {
            const float mw0 = mlb[(v * 8 + h0) * 2], mw1 = mlb[(v * 8 + h1) * 2];
            sc0[v] = mw0 == -INFINITY ? 0.f : ex2(mw0 - ms0);
            sc1[v] = mw1 == -INFINITY ? 0.f : ex2(mw1 - ms1);
            if (v == 0) {
                ls0 = sc0[0] * mlb[h0 * 2 + 1];
                ls1 = sc1[0] * mlb[h1 * 2 + 1];
            } else {
                ls0 += sc0[v] * mlb[(v * 8 + h0) * 2 + 1];
                ls1 += sc1[v] * mlb[(v * 8 + h1) * 2 + 1];
            }
        }
        int iu, isp, ins;   // found again here rather than kept live through the item
        kivi_unit_split(p, item, iu, isp, ins);
        const bool single = ins == 1;
        const size_t pi0 = ((size_t)(iu - p.full_units) * p.splits + isp) * p.g;
        const int hs[2] = {h0, h1};
        const float lss[2] = {ls0, ls1}, mss[2] = {ms0, ms1};
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m / OWN != warp)
                continue;
            const float *src = ob + warp * (NCW - 1) * 8 * OSTR + (m - warp * OWN) * 16;
            float o[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int v = 0; v < NCW; ++v) {
                float x[4];
                if (v == warp) {
                    x[0] = acc[m][0];
                    x[1] = acc[m][1];
                    x[2] = acc[m][2];
                    x[3] = acc[m][3];
                } else {
                    const float *sv = src + (v < warp ? v : v - 1) * 8 * OSTR;
                    x[0] = sv[h0 * OSTR + r];
                    x[1] = sv[h1 * OSTR + r];
                    x[2] = sv[h0 * OSTR + r + 8];
                    x[3] = sv[h1 * OSTR + r + 8];
                }
                if (v == 0) {
                    o[0] = x[0] * sc0[0];
                    o[1] = x[1] * sc1[0];
                    o[2] = x[2] * sc0[0];
                    o[3] = x[3] * sc1[0];
                } else {
                    o[0] += sc0[v] * x[0];
                    o[1] += sc1[v] * x[1];
                    o[2] += sc0[v] * x[2];
                    o[3] += sc1[v] * x[3];
                }
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int h = hs[e];
                if (h >= p.g)
                    continue;
                if (single) {
                    const float inv = lss[e] > 0.f ? 1.f / lss[e] : 0.f;
                    uint16_t *orow = p.o + ((size_t)b * p.Hq + hk * p.g + h) * D;
                    orow[16 * m + r] = __half_as_ushort(__float2half_rn(o[e] * inv));
                    orow[16 * m + r + 8] = __half_as_ushort(__float2half_rn(o[2 + e] * inv));
                } else {
                    float *po = p.part_o + (pi0 + h) * D;
                    po[16 * m + r] = o[e];
                    po[16 * m + r + 8] = o[2 + e];
                }
            }
        }
        if (warp == 0 && r == 0) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int h = hs[e];
                if (h >= p.g)
                    continue;
                if (single) {
                    if (p.lse)
                        p.lse[(size_t)b * p.Hq + hk * p.g + h] =
                            lss[e] > 0.f ? (mss[e] + __log2f(lss[e])) * LN2 : -INFINITY;
                } else {
                    p.part_ml[2 * (pi0 + h)] = lss[e] > 0.f ? mss[e] : -INFINITY;
                    p.part_ml[2 * (pi0 + h) + 1] = lss[e];
                }
            }
        }
    }
    }   // items
}

template <int D, int BITS, bool GEAR>
cudaError_t launch_kivi_impl(const KiviAttendLaunch &a, const KiviParams &kp, cudaStream_t s)
{
    using Cfg = KiviCfg<D, BITS, GEAR>;
    // the residual rings as [B * Hkv * (R + 32), D] fp16, one box = RS ring slots
    CUtensorMap tk, tv;
    const uint64_t rows = (uint64_t)a.B * a.Hkv * kp.CR;
    if (!encode_tmap_2d_f16(&tk, a.k_res, D, rows, 64, Cfg::RS) ||
        !encode_tmap_2d_f16(&tv, a.v_res, D, rows, 64, Cfg::RS))
        return cudaErrorInvalidValue;
    const void *fn = reinterpret_cast<const void *>(k_attend_kivi<D, BITS, GEAR>);
    const cudaError_t e = set_smem_once(fn, Cfg::SMEM);
    if (e != cudaSuccess)
        return e;
    const int resident = resident_ctas(fn, NTHREADS, Cfg::SMEM);
    const int grid = kp.n_items < resident ? kp.n_items : resident;
    if (grid <= 0)
        return cudaSuccess;
    k_attend_kivi<D, BITS, GEAR><<<grid, NTHREADS, Cfg::SMEM, s>>>(tk, tv, kp);
    return cudaGetLastError();
}

template <int D, int BITS>
cudaError_t launch_kivi_bits(const KiviAttendLaunch &a, const KiviParams &kp, cudaStream_t s)
{
    static_assert(KiviCfg<128, BITS, true>::SIDE == 976 && KiviCfg<64, BITS, true>::SIDE == 560,
                  "GEAR side block size");
    return kp.kg ? launch_kivi_impl<D, BITS, true>(a, kp, s)
                 : launch_kivi_impl<D, BITS, false>(a, kp, s);
}

} // namespace

cudaError_t launch_attend_kivi(const KiviAttendLaunch &a, cudaStream_t s)
{
    const int CR = a.R + KIVI_G;
    KiviParams kp{};
    kp.Hq = a.Hq;
    kp.Hkv = a.Hkv;
    kp.g = a.Hq / a.Hkv;
    kp.Cq = a.Cq;
    kp.R = a.R;
    kp.CR = CR;
    kp.splits = a.splits;
    kp.qtiles_per_split = a.tiles_per_split;
    kp.q = a.q;
    kp.o = a.o;
    kp.lse = a.lse;
    kp.kb = a.kb;
    kp.vb = a.vb;
    kp.kg = a.kg;
    kp.vg = a.vg;
    kp.blocks = GroupBlocks{a.block_table, a.Cq / KIVI_G, a.num_pages,
                            (int)kvc_kivi_block_bytes(a.D, a.bits)};
    kp.len = a.len;
    kp.part_o = a.splits > 1 ? a.part_o : nullptr;
    kp.part_ml = a.splits > 1 ? a.part_ml : nullptr;
    kp.scale = a.scale;
    kp.scale_log2 = a.scale * LOG2E;
    kp.status = dev_status_ptr();
    const int units = a.B * a.Hkv;
    kp.full_units = a.splits > 1 ? a.full_units : units;
    kp.n_items = kp.full_units + (units - kp.full_units) * a.splits;
    cudaError_t e;
    if (a.D == 128)
        e = a.bits == 4 ? launch_kivi_bits<128, 4>(a, kp, s) : launch_kivi_bits<128, 2>(a, kp, s);
    else
        e = a.bits == 4 ? launch_kivi_bits<64, 4>(a, kp, s) : launch_kivi_bits<64, 2>(a, kp, s);
    if (e != cudaSuccess || a.splits == 1)
        return e;
    return launch_combine(a.B, a.Hq, a.Hkv, a.D, a.splits, a.full_units, units - a.full_units,
                          a.part_o, a.part_ml, a.o, a.lse, s);
}

} // namespace kvc
