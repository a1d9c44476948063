// h2o_prefill_tc.cu -- the H2O prefill score pass on the 5th-generation tensor
// cores (tcgen05.mma, accumulators in TMEM).
//
// The heavy-hitter score of prompt token j is the attention it receives from
// every later prompt row, summed over the query heads of its KV head
// ("Rethinking KV Cache Compression" guide, §16 "局限与最终结论": flash attention
// never materialises the probabilities, so scoring needs an extra pass):
//   pass 1  lse_i = log2 sum_{j <= i} 2^(s_ij)          (s = scale log2e q_i . k_j)
//   pass 2  score_j = sum_{h in group} sum_{i >= j} 2^(s_ij - lse_i)
// Pass 1 stores -lse_i; pass 2 brings each query tile's 128 values into a small
// shared-memory ring with the tile, so its epilogue reads them from there.  A
// caller that already holds the rows' normalisers (a causal flash-attention
// forward over the prompt computes them) passes them in and skips pass 1: then
// only the extra pass of the guide's statement runs.
//
// A work item is one 128-row "stationary" tile held in shared memory -- a query
// tile in pass 1, a key tile in pass 2 -- against every 128-row tile of the
// other operand it meets under the causal mask, streamed through a TMA ring.
// Causal items are paired (t, nt-1-t) so all pairs cost the same; the CTAs are
// persistent and walk the pairs round-robin.  One thread issues tcgen05.mma
// (M = N = 128, fp16 in, fp32 out) into one of two TMEM accumulators, so the
// next product runs while eight epilogue warps read the previous one.  TMEM
// lane r is row r of the product (a query row in pass 1, a key row in pass 2);
// the two warps of a lane quarter take one half of the 128 columns each, keep a
// partial row state (online max / sum, or a probability sum) and merge it at
// the end of the item.  Each 32-column chunk is classified per warp as inside
// the causal window, outside it (skipped) or cut by it (masked), so only the
// diagonal and the ragged tail pay for masks; the arithmetic runs on packed
// fp32 pairs.
#include "kvc_device.cuh"
#include "kvc_internal.h"

#include <math.h>

namespace kvc {

namespace {

constexpr int TT = 128;                  // rows of every tile
constexpr int NQ = 4;                    // TMEM lane quarters
constexpr int NEPI = 2 * NQ;             // epilogue warps: two column halves per quarter
constexpr int NTHR = (2 + NEPI) * 32;    // warp 0: TMA producer, warp 1: MMA issuer
constexpr int NS = 2;                    // streaming stages
constexpr int NL = 4;                    // pass 2: -lse slots of 128 floats
constexpr int NI = 2;                    // slots of the pair feed
constexpr int TMEM_COLS = 2 * TT;        // two fp32 accumulators of 128 columns
constexpr int CTAS_PER_SM = 2;
constexpr float LOG2E = 1.4426950408889634f;

template <int D> struct TcCfg {
    static constexpr int NBOX = D / 64;
    static constexpr int BOX_BYTES = TT * 128;
    static constexpr int TILE_BYTES = NBOX * BOX_BYTES;
    static constexpr int LSE_BYTES = NL * TT * 4;
    static constexpr int MERGE_BYTES = NQ * 32 * 8;          // row state of the second column half
    static constexpr int SMEM_USED = (1 + NS) * TILE_BYTES + LSE_BYTES + MERGE_BYTES + 512 + 1024;
    // at most two CTAs per SM: each holds half of the SM's 512 TMEM columns
    static constexpr int SMEM = SMEM_USED > 80 * 1024 ? SMEM_USED : 80 * 1024;
    static constexpr uint32_t IDESC = idesc_f16_f32(TT, TT);
};

struct TcParams {
    int Hq, Hkv, g, L, Lpad, kp_cap, C, nt, npairs, n_work;
    float *nlse;        // [B*Hq, Lpad]: -lse of every prompt row (pass 1 writes, pass 2 reads)
    int *work_ctr;      // pairs handed out beyond each CTA's first (zero at launch)
    float *scores;
    float scale_log2;
    int *status;
};

// Work is handed out in pairs: pair w covers tiles w % npairs and
// nt - 1 - w % npairs (one tile when they coincide) of the (head or unit)
// w / npairs, so every pair costs the same.  A CTA starts with pair blockIdx.x
// and then takes the next unclaimed pair from a global counter, so the two
// CTAs that share an SM (which progress at different rates) finish together.
__device__ __forceinline__ int pair_items(const TcParams &p, int w)
{
    const int pair = w % p.npairs;
    return pair != p.nt - 1 - pair ? 2 : 1;
}

// Walks the stream tiles of an item on tile t in order: pass 1 key tiles
// qt = 0 .. t; pass 2 query tiles qt = t .. nt-1 of group head hh = 0, then of
// head 1, and so on.
template <int PASS> struct StreamWalk {
    int hh, qt;
    __device__ explicit StreamWalk(int t) : hh(0), qt(PASS == 1 ? 0 : t) {}
    __device__ void next(const TcParams &p, int t)
    {
        if (PASS == 1) {
            ++qt;
        } else if (++qt == p.nt) {
            qt = t;
            ++hh;
        }
    }
};

template <int PASS> __device__ __forceinline__ int n_stream(const TcParams &p, int t)
{
    return PASS == 1 ? t + 1 : p.g * (p.nt - t);
}

// 2^x as an ordered statement: the exponentials of one chunk are issued before
// the next chunk's TMEM load, so a thread never holds two chunks at once.
__device__ __forceinline__ float ex2o(float x)
{
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

enum ChunkClass { CH_NONE = 0, CH_FULL = 1, CH_PART = 2 };

// Pass 1: fold 32 key columns j0 + c into the online (m, l) of query row gi.
template <bool MASK>
__device__ __forceinline__ void p1_chunk(const float *v, int j0, int gi, int L, float scale,
                                         float &m, float &l)
{
    float x[32];
#pragma unroll
    for (int c = 0; c < 32; ++c)
        x[c] = (!MASK || (j0 + c <= gi && j0 + c < L)) ? v[c] : -INFINITY;
    float c0 = fmax3f(x[0], x[1], x[2]), c1 = fmax3f(x[8], x[9], x[10]);
    float c2 = fmax3f(x[16], x[17], x[18]), c3 = fmax3f(x[24], x[25], x[26]);
#pragma unroll
    for (int k = 3; k < 7; k += 2) {
        c0 = fmax3f(c0, x[k], x[k + 1]);
        c1 = fmax3f(c1, x[8 + k], x[9 + k]);
        c2 = fmax3f(c2, x[16 + k], x[17 + k]);
        c3 = fmax3f(c3, x[24 + k], x[25 + k]);
    }
    const float mx = fmaxf(fmax3f(c0, c1, x[7]), fmax3f(c2, c3, fmax3f(x[15], x[23], x[31])));
    const float mn = fmaxf(m, mx * scale);
    const float ref = mn == -INFINITY ? 0.f : mn;
    const float2 sc2 = make_float2(scale, scale), nr2 = make_float2(-ref, -ref);
    float2 a0 = make_float2(0.f, 0.f), a1 = a0;
#pragma unroll
    for (int c = 0; c < 32; c += 4) {
        const float2 y0 = ffma2(make_float2(x[c], x[c + 1]), sc2, nr2);
        const float2 y1 = ffma2(make_float2(x[c + 2], x[c + 3]), sc2, nr2);
        a0 = fadd2(a0, make_float2(ex2o(y0.x), ex2o(y0.y)));
        a1 = fadd2(a1, make_float2(ex2o(y1.x), ex2o(y1.y)));
    }
    const float2 a = fadd2(a0, a1);
    l = l * ex2o(m - ref) + (a.x + a.y);
    m = mn;
}

// Pass 2: sum over 32 query columns i0 + c of 2^(s scale - lse_i) for key row gi;
// nlse holds -lse_i of those columns (-inf past the prompt, so only the causal
// diagonal needs a mask).
template <bool MASK>
__device__ __forceinline__ float p2_chunk(const float *v, const float *nlse, int i0, int gi, int L,
                                          float scale)
{
    const float2 sc2 = make_float2(scale, scale);
    float2 a0 = make_float2(0.f, 0.f), a1 = a0;
#pragma unroll
    for (int c = 0; c < 32; c += 4) {
        const float4 nl = *reinterpret_cast<const float4 *>(nlse + c);
        const float2 y0 = ffma2(make_float2(v[c], v[c + 1]), sc2, make_float2(nl.x, nl.y));
        const float2 y1 = ffma2(make_float2(v[c + 2], v[c + 3]), sc2, make_float2(nl.z, nl.w));
        float e[4] = {ex2o(y0.x), ex2o(y0.y), ex2o(y1.x), ex2o(y1.y)};
        if (MASK) {
#pragma unroll
            for (int u = 0; u < 4; ++u)
                e[u] = i0 + c + u >= gi ? e[u] : 0.f;
        }
        a0 = fadd2(a0, make_float2(e[0], e[1]));
        a1 = fadd2(a1, make_float2(e[2], e[3]));
    }
    const float2 a = fadd2(a0, a1);
    return a.x + a.y;
}

// Fold this warp's two 32-column chunks of one accumulator tile (TMEM columns
// taddr .. taddr + 63 of the warp's lanes) into the thread's row state, handing
// the accumulator back once both chunks are in registers.  Returns the pass-2
// sum of the chunks (0 in pass 1).
template <int PASS>
__device__ __forceinline__ float fold_tile(uint32_t taddr, uint64_t *acc_empty, int cls0, int cls1,
                                           int col0, int gi, const TcParams &p, const float *nlse,
                                           float &m, float &l)
{
    float tile_sum = 0.f;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int cls = k == 0 ? cls0 : cls1;
        float v[32];
        if (cls != CH_NONE)
            tmem_ld32(taddr + 32 * k, v);
        if (k == 1) {
            tc_fence_before();
            __syncwarp();
            mbar_arrive_warp(acc_empty);
        }
        const int c0 = col0 + 32 * k;
        if (PASS == 1) {
            if (cls == CH_FULL)
                p1_chunk<false>(v, c0, gi, p.L, p.scale_log2, m, l);
            else if (cls == CH_PART)
                p1_chunk<true>(v, c0, gi, p.L, p.scale_log2, m, l);
        } else {
            if (cls == CH_FULL)
                tile_sum += p2_chunk<false>(v, nlse + 32 * k, c0, gi, p.L, p.scale_log2);
            else if (cls == CH_PART)
                tile_sum += p2_chunk<true>(v, nlse + 32 * k, c0, gi, p.L, p.scale_log2);
        }
    }
    return tile_sum;
}

template <int D, int PASS>
__global__ void __launch_bounds__(NTHR, CTAS_PER_SM)
    k_prefill_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const TcParams p)
{
    using Cfg = TcCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_align1024(smem_raw);
    uint8_t *stat = smem;                                   // stationary tile
    uint8_t *ring = smem + Cfg::TILE_BYTES;                 // NS streaming tiles
    float *lse_buf = reinterpret_cast<float *>(smem + (1 + NS) * Cfg::TILE_BYTES);
    double *merge = reinterpret_cast<double *>(smem + (1 + NS) * Cfg::TILE_BYTES + Cfg::LSE_BYTES);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (1 + NS) * Cfg::TILE_BYTES + Cfg::LSE_BYTES +
                                                  Cfg::MERGE_BYTES);
    uint64_t *s_full = bars, *s_empty = bars + NS;
    uint64_t *acc_full = bars + 2 * NS, *acc_empty = bars + 2 * NS + 2;
    uint64_t *stat_full = bars + 2 * NS + 4, *stat_empty = bars + 2 * NS + 5;
    uint64_t *mma_done = bars + 2 * NS + 6;
    uint64_t *mrg_full = bars + 2 * NS + 7, *mrg_empty = bars + 2 * NS + 7 + NQ;
    uint64_t *l_full = bars + 2 * NS + 7 + 2 * NQ, *l_empty = l_full + NL;
    uint64_t *it_full = l_empty + NL, *it_empty = it_full + NI;
    __shared__ uint32_t s_tmem;
    __shared__ int s_item[NI];
    __shared__ int s_abort;
    volatile int *abort = &s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // (b, hk) and the head (pass 1) / KV unit (pass 2) of an item's outer index
    auto decode = [&](int outer, int &b, int &hk, int &bh, int &unit) {
        if (PASS == 1) {
            bh = outer;
            b = bh / p.Hq;
            hk = (bh % p.Hq) / p.g;
            unit = b * p.Hkv + hk;
        } else {
            bh = 0;
            unit = outer;
            b = unit / p.Hkv;
            hk = unit % p.Hkv;
        }
    };

    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int i = 0; i < NS; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&acc_full[i], 1);
            mbar_init(&acc_empty[i], NEPI);
        }
        mbar_init(stat_full, 1);
        mbar_init(stat_empty, 1);
        mbar_init(mma_done, 1);
        for (int q = 0; q < NQ; ++q) {
            mbar_init(&mrg_full[q], 32);
            mbar_init(&mrg_empty[q], 32);
        }
        for (int i = 0; i < NL; ++i) {
            mbar_init(&l_full[i], 1);
            mbar_init(&l_empty[i], NEPI);
        }
        for (int i = 0; i < NI; ++i) {
            mbar_init(&it_full[i], 1);
            mbar_init(&it_empty[i], 1 + NEPI);   // the MMA thread and every epilogue warp
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&s_tmem, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    // The pair feed: the producer publishes the k-th pair in slot k % NI; the MMA
    // thread and the epilogue warps read the pairs in the same order.  A pair
    // index >= n_work ends the walk.
    auto feed_put = [&](int k, int w) -> bool {
        const int slot = k % NI;
        if (k >= NI && !mbar_sleep_or_abort(&it_empty[slot], ((k / NI) & 1) ^ 1, abort))
            return false;
        s_item[slot] = w;
        mbar_arrive(&it_full[slot]);
        return true;
    };
    // consumers: the next item (outer index, stationary tile t) of the feed
    struct FeedCursor {
        int k = 0, w = 0, h = 0, nh = 0;
    };
    auto feed_next = [&](FeedCursor &c, int &outer, int &t, bool whole_warp) -> bool {
        if (c.h >= c.nh) {
            const int slot = c.k % NI;
            bool got = mbar_sleep_or_abort(&it_full[slot], (c.k / NI) & 1, abort);
            if (whole_warp)
                got = __all_sync(0xffffffffu, got);
            if (!got)
                return false;
            c.w = *reinterpret_cast<volatile int *>(&s_item[slot]);
            if (whole_warp)
                __syncwarp();
            if (!whole_warp || lane == 0)
                mbar_arrive(&it_empty[slot]);
            ++c.k;
            if (c.w >= p.n_work)
                return false;
            c.h = 0;
            c.nh = pair_items(p, c.w);
        }
        const int pair = c.w % p.npairs;
        outer = c.w / p.npairs;
        t = c.h == 0 ? pair : p.nt - 1 - pair;
        ++c.h;
        return true;
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&tmQ);
            prefetch_tmap(&tmK);
            int it = 0, n_stat = 0, outer, t;
            bool ok = true;
            int fk = 0, fw = blockIdx.x, fh = 0, fnh = 0;   // pairs published, current pair
            while (ok) {
                if (fh >= fnh) {
                    if (fk > 0)
                        fw = gridDim.x + atomicAdd(p.work_ctr, 1);
                    if (!feed_put(fk++, fw) || fw >= p.n_work)
                        break;
                    fh = 0;
                    fnh = pair_items(p, fw);
                }
                outer = fw / p.npairs;
                t = fh == 0 ? fw % p.npairs : p.nt - 1 - fw % p.npairs;
                ++fh;
                int b, hk, bh, unit;
                decode(outer, b, hk, bh, unit);
                if (n_stat > 0 && !mbar_sleep_or_abort(stat_empty, (n_stat - 1) & 1, abort))
                    break;
                ++n_stat;
                mbar_arrive_expect_tx(stat_full, Cfg::TILE_BYTES);
#pragma unroll
                for (int j = 0; j < Cfg::NBOX; ++j) {
                    if (PASS == 1)
                        tma_load_2d(stat + j * Cfg::BOX_BYTES, &tmQ, stat_full, 64 * j,
                                    bh * p.L + t * TT);
                    else
                        tma_load_2d(stat + j * Cfg::BOX_BYTES, &tmK, stat_full, 64 * j,
                                    unit * p.kp_cap + t * TT);
                }
                const int ns = n_stream<PASS>(p, t);
                StreamWalk<PASS> sp(t);
                for (int s = 0; s < ns; ++s, ++it, sp.next(p, t)) {
                    const int st = it % NS;
                    if (it >= NS && !mbar_sleep_or_abort(&s_empty[st], ((it / NS) & 1) ^ 1, abort)) {
                        ok = false;
                        break;
                    }
                    uint8_t *dst = ring + st * Cfg::TILE_BYTES;
                    if (PASS == 2) {
                        const int ls = it % NL;
                        if (it >= NL &&
                            !mbar_sleep_or_abort(&l_empty[ls], ((it / NL) & 1) ^ 1, abort)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&l_full[ls], TT * 4);
                        bulk_load(lse_buf + ls * TT,
                                  p.nlse + (size_t)(b * p.Hq + hk * p.g + sp.hh) * p.Lpad + sp.qt * TT,
                                  TT * 4, &l_full[ls]);
                    }
                    mbar_arrive_expect_tx(&s_full[st], Cfg::TILE_BYTES);
#pragma unroll
                    for (int j = 0; j < Cfg::NBOX; ++j) {
                        if (PASS == 1)
                            tma_load_2d(dst + j * Cfg::BOX_BYTES, &tmK, &s_full[st], 64 * j,
                                        unit * p.kp_cap + sp.qt * TT);
                        else
                            tma_load_2d(dst + j * Cfg::BOX_BYTES, &tmQ, &s_full[st], 64 * j,
                                        (b * p.Hq + hk * p.g + sp.hh) * p.L + sp.qt * TT);
                    }
                }
            }
            // Every copy has landed before the CTA leaves.  Normally the MMA
            // thread consumed them all; after a timeout this bounds the wait.
            for (int i = it > NS ? it - NS : 0; i < it; ++i)
                mbar_wait(&s_full[i % NS], (i / NS) & 1);
            if (PASS == 2)
                for (int i = it > NL ? it - NL : 0; i < it; ++i)
                    mbar_wait(&l_full[i % NL], (i / NL) & 1);
            if (n_stat > 0)
                mbar_wait(stat_full, (n_stat - 1) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int it = 0, tc = 0, n_item = 0, outer, t;
            bool ok = true;
            FeedCursor fc;
            for (; ok && feed_next(fc, outer, t, false); ++n_item) {
                if (!mbar_sleep_or_abort(stat_full, n_item & 1, abort))
                    break;
                tc_fence_after();
                const uint32_t sbase = smem_u32(stat);
                const int ns = n_stream<PASS>(p, t);
                for (int s = 0; s < ns; ++s, ++it, ++tc) {
                    const int st = it % NS, buf = tc & 1;
                    if (!mbar_sleep_or_abort(&s_full[st], (it / NS) & 1, abort) ||
                        (tc >= 2 &&
                         !mbar_sleep_or_abort(&acc_empty[buf], ((tc / 2) & 1) ^ 1, abort))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t rbase = smem_u32(ring + st * Cfg::TILE_BYTES);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * Cfg::BOX_BYTES + (kk & 3) * 32;
                        umma_f16(tmem + buf * TT, sdesc_k_sw128(sbase + off),
                                 sdesc_k_sw128(rbase + off), Cfg::IDESC, kk > 0 ? 1u : 0u);
                    }
                    umma_commit(&s_empty[st]);
                    umma_commit(&acc_full[buf]);
                }
                umma_commit(stat_empty);
            }
            // every product this thread issued has finished before TMEM is released
            umma_commit(mma_done);
            mbar_wait(mma_done, 0);
        }
    } else {
        // ------------------------------------------------ epilogue warps
        const int e = warp - 2;
        const int quarter = warp & 3;              // TMEM lanes [32 quarter, 32 quarter + 32)
        const int half = e / NQ;                   // columns [64 half, 64 half + 64)
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * quarter) << 16) + 64 * half;
        int tc = 0, n_item = 0, outer, t;
        bool ok = true;
        FeedCursor fc;
        for (; ok && feed_next(fc, outer, t, true); ++n_item) {
            int b, hk, bh, unit;
            decode(outer, b, hk, bh, unit);
            const int ns = n_stream<PASS>(p, t);
            const int r0 = t * TT + 32 * quarter;   // first row of this warp
            const int gi = r0 + lane;               // this thread's query (1) / key (2) row
            float m = -INFINITY, l = 0.f;           // pass 1
            double acc = 0.0;                       // pass 2
            float run = 0.f;
            StreamWalk<PASS> sp(t);
            for (int s = 0; s < ns; ++s, ++tc, sp.next(p, t)) {
                const int buf = tc & 1;
                const int ls = tc % NL;
                // pass 2: the tile's -lse has landed in slot ls; then the
                // accumulator (every lane acquires both)
                const bool got =
                    (PASS == 1 || mbar_wait_or_abort(&l_full[ls], (tc / NL) & 1, abort)) &&
                    mbar_wait_or_abort(&acc_full[buf], (tc / 2) & 1, abort);
                if (!__all_sync(0xffffffffu, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // Tiles off the diagonal lie wholly inside the causal window;
                // otherwise each of this warp's 32-column chunks is classified.
                const int col0 = sp.qt * TT + 64 * half;   // first key (1) / query (2) column
                const float *nl = lse_buf + ls * TT + 64 * half;
                const bool inside = PASS == 1 ? sp.qt < t : sp.qt > t;
                float tile_sum;
                if (inside) {
                    tile_sum = fold_tile<PASS>(lane_addr + buf * TT, &acc_empty[buf], CH_FULL,
                                               CH_FULL, col0, gi, p, nl, m, l);
                } else {
                    int cls[2];
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const int c0 = col0 + 32 * k;
                        if (PASS == 1)
                            cls[k] = (c0 >= p.L || c0 > r0 + 31)          ? CH_NONE
                                     : (c0 + 31 <= r0 && c0 + 31 < p.L)   ? CH_FULL
                                                                          : CH_PART;
                        else
                            cls[k] = (c0 >= p.L || c0 + 31 < r0) ? CH_NONE
                                     : c0 >= r0 + 31                 ? CH_FULL
                                                                     : CH_PART;
                    }
                    tile_sum = fold_tile<PASS>(lane_addr + buf * TT, &acc_empty[buf], cls[0],
                                               cls[1], col0, gi, p, nl, m, l);
                }
                if (PASS == 2) {
                    // fp32 over the tiles of one query head, fp64 across heads
                    run += tile_sum;
                    if (sp.qt == p.nt - 1) {
                        acc += (double)run;
                        run = 0.f;
                    }
                    __syncwarp();   // every lane has read the slot
                    mbar_arrive_warp(&l_empty[ls]);
                }
            }
            if (!ok)
                break;
            // merge the two column halves of each row: the second half hands its
            // state over through shared memory (bounded waits both ways)
            double *mq = merge + quarter * 32;
            if (half == 1) {
                const bool drained = n_item == 0 ||
                                  mbar_sleep_or_abort(&mrg_empty[quarter], (n_item - 1) & 1, abort);
                if (!__all_sync(0xffffffffu, drained))
                    break;
                if (PASS == 1)
                    reinterpret_cast<float2 *>(mq)[lane] = make_float2(m, l);
                else
                    mq[lane] = acc;
                mbar_arrive(&mrg_full[quarter]);
            } else {
                const bool ready = mbar_sleep_or_abort(&mrg_full[quarter], n_item & 1, abort);
                if (!__all_sync(0xffffffffu, ready))
                    break;
                double other = mq[lane];
                mbar_arrive(&mrg_empty[quarter]);
                if (PASS == 1) {
                    // rows of the last tile past L get -lse = -inf, so their
                    // columns add 2^-inf = 0 in pass 2 without a mask
                    const float2 o = *reinterpret_cast<const float2 *>(&other);
                    const float mm = fmaxf(m, o.x);
                    const float ll = l * ex2o(m - mm) + o.y * ex2o(o.x - mm);
                    p.nlse[(size_t)bh * p.Lpad + gi] = gi < p.L ? -(mm + __log2f(ll)) : -INFINITY;
                } else if (gi < p.L) {
                    p.scores[(size_t)unit * p.C + gi] = (float)(acc + other);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
    if (threadIdx.x == 0 && *abort)
        flag_error(p.status, DEV_TIMEOUT);
}

template <int D, int PASS>
cudaError_t launch_tc(const CUtensorMap &tq, const CUtensorMap &tk, const TcParams &tp,
                      cudaStream_t s)
{
    using Cfg = TcCfg<D>;
    const cudaError_t e =
        set_smem_once(reinterpret_cast<const void *>(k_prefill_tc<D, PASS>), Cfg::SMEM);
    if (e != cudaSuccess)
        return e;
    const int cap = CTAS_PER_SM * sm_count();
    const int grid = tp.n_work < cap ? tp.n_work : cap;
    k_prefill_tc<D, PASS><<<grid, NTHR, Cfg::SMEM, s>>>(tq, tk, tp);
    return cudaGetLastError();
}

// -lse rows for pass 2 from normalisers the caller already has (the natural-log
// log-sum-exp of each prompt row, as a causal flash-attention forward returns
// it): -lse * log2e in the log2 domain of pass 1, -inf on the padding rows.
__global__ void k_nlse_from_lse(const float *__restrict__ lse, float *__restrict__ nlse,
                                long long rows, int L, int Lpad)
{
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= rows * Lpad)
        return;
    const long long r = i / Lpad;
    const int c = (int)(i - r * Lpad);
    nlse[i] = c < L ? -lse[r * L + c] * LOG2E : -INFINITY;
}

template <int D> cudaError_t prefill_tc_impl(const kvc_h2o_args &a, float *lse_ws, cudaStream_t s)
{
    TcParams tp{};
    tp.Hq = a.Hq;
    tp.Hkv = a.Hkv;
    tp.g = a.Hq / a.Hkv;
    tp.L = a.L;
    tp.nt = (a.L + TT - 1) / TT;
    tp.Lpad = tp.nt * TT;
    tp.npairs = (tp.nt + 1) / 2;
    tp.kp_cap = a.kp_cap;
    tp.C = a.C;
    tp.nlse = lse_ws;
    // the two passes' pair counters follow the -lse rows in the workspace
    int *ctr = reinterpret_cast<int *>(lse_ws + (size_t)a.B * a.Hq * tp.Lpad);
    cudaError_t e0 = cudaMemsetAsync(ctr, 0, 2 * sizeof(int), s);
    if (e0 != cudaSuccess)
        return e0;
    tp.scores = a.scores;
    const float scale = a.softmax_scale > 0.f ? a.softmax_scale : 1.0f / sqrtf((float)a.D);
    tp.scale_log2 = scale * LOG2E;
    tp.status = dev_status_ptr();
    CUtensorMap tq, tk;
    if (!encode_tmap_2d_f16(&tq, a.qp, D, (uint64_t)a.B * a.Hq * a.L, 64, TT) ||
        !encode_tmap_2d_f16(&tk, a.kp, D, (uint64_t)a.B * a.Hkv * a.kp_cap, 64, TT))
        return cudaErrorInvalidValue;
    if (a.lse) {   // the rows' normalisers are given: only the column-sum pass runs
        const long long rows = (long long)a.B * a.Hq, total = rows * tp.Lpad;
        k_nlse_from_lse<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(a.lse, lse_ws, rows, a.L,
                                                                        tp.Lpad);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess)
            return e;
    } else {
        tp.n_work = a.B * a.Hq * tp.npairs;
        tp.work_ctr = ctr;
        const cudaError_t e = launch_tc<D, 1>(tq, tk, tp, s);
        if (e != cudaSuccess)
            return e;
    }
    tp.n_work = a.B * a.Hkv * tp.npairs;
    tp.work_ctr = ctr + 1;
    return launch_tc<D, 2>(tq, tk, tp, s);
}

} // namespace

cudaError_t launch_h2o_prefill(const kvc_h2o_args &a, float *lse_ws, cudaStream_t s)
{
    return a.D == 128 ? prefill_tc_impl<128>(a, lse_ws, s) : prefill_tc_impl<64>(a, lse_ws, s);
}

} // namespace kvc
