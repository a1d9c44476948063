// evict.cu -- keep-set selection and in-place compaction of slot caches.
//
// One CTA per (sequence, KV head) unit (one warp per unit for caches of at
// most 1024 slots, the decode-sized H2O and StreamingLLM caches):
//   1. decide the keep set
//        H2O    ("Rethinking KV Cache Compression" guide, §2 and §16 "4 种方法
//               逐步执行"): the recent window pos >= T - n_recent, plus the
//               n_heavy other slots with the largest accumulated scores (ties:
//               lower position) -- a radix select of the n_heavy-th smallest
//               composite key (descending-score bits << 32 | pos);
//        Stream (same page): pos < n_sink or pos >= T - n_recent, closed form;
//        Random ("KV Cache 驱逐实战", section "参考实现"): prompt slots stay;
//               n_keep = max(1, int(n_cand * keep_ratio)) candidates with the
//               smallest 64-bit Philox4x32-10 keys (ties: lower position),
//               drawn independently in every head;
//   2. compact: with n' kept slots, the k-th hole in [0, n') receives the k-th
//      kept slot of [n', n) (mark and compact, "Practical Online KV Cache
//      Compaction for LLM Agents", §4.2; the pos array is the logical ->
//      physical map).  Sources and destinations never overlap, so the moves
//      run in parallel; K, V, pos (and H2O scores) move together.
#include "kvc_device.cuh"
#include "kvc_internal.h"

namespace kvc {

namespace {

constexpr int ETHREADS = 256;
constexpr int NWARPS = ETHREADS / 32;
constexpr int HOLE_CAP = 2048;   // hole/tail pairs handled per compaction round
constexpr int MAX_SLOTS = 65536; // slot capacity the keep bitmask covers

struct EvictParams {
    int Hkv, D, C;
    uint16_t *K, *V;
    int32_t *pos, *n;
    const int32_t *seqlen;
    float *scores;
    int n_heavy, n_recent, n_sink, prompt_len;
    int trigger;        // H2O: units with n < trigger are left unchanged
    SlotRows rows;      // K / V rows of each slot (dense or paged)
    double keep_ratio;
    uint32_t seed_lo, seed_hi, epoch;
    int *status;
};

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of
// (c0,c1,c2,c3) -> (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)),
// M0 = 0xD2511F53, M1 = 0xCD9E8D57, key bumped by (0x9E3779B9, 0xBB67AE85).
__device__ __forceinline__ uint64_t philox_key(uint32_t k0, uint32_t k1, uint32_t c0, uint32_t c1,
                                               uint32_t c2, uint32_t c3)
{
#pragma unroll
    for (int rnd = 0; rnd < 10; ++rnd) {
        if (rnd > 0) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
        const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
    }
    return ((uint64_t)c0 << 32) | c1;
}

struct Shared {
    uint32_t hist[256];
    int warp_tot[NWARPS];
    int bcast[4];
    uint32_t keep[MAX_SLOTS / 32];
    int hole[HOLE_CAP];
    int mv_src[HOLE_CAP];
    int mv_dst[HOLE_CAP];
};

// Exclusive block-wide scan of one int per thread; returns the exclusive
// prefix and sets *total.  All threads must call it.
__device__ __forceinline__ int block_scan(int v, int *total, Shared &sh)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off)
            x += y;
    }
    if (lane == 31)
        sh.warp_tot[warp] = x;
    __syncthreads();
    int base = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < NWARPS; ++w) {
        if (w < warp)
            base += sh.warp_tot[w];
        tot += sh.warp_tot[w];
    }
    __syncthreads();
    *total = tot;
    return base + x - v;
}

__device__ __forceinline__ int block_count(bool pred, Shared &sh)
{
    int tot;
    block_scan(pred ? 1 : 0, &tot, sh);
    return tot;
}

// k-th smallest (1-based) of key(j) over slots j < n with filt(j), radix 8 bits
// at a time from the top of `nbits`.  Returns the key value; *rank_left gets
// how many slots equal to it are within the first k.
template <typename KeyFn, typename FiltFn>
__device__ uint64_t radix_select(int n, int k, int nbits, KeyFn key, FiltFn filt, int *rank_left,
                                 Shared &sh)
{
    uint64_t prefix = 0, mask = 0;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int shift = nbits - 8; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += ETHREADS)
            sh.hist[i] = 0;
        __syncthreads();
        for (int j = threadIdx.x; j < n; j += ETHREADS) {
            if (!filt(j))
                continue;
            const uint64_t kk = key(j);
            if ((kk & mask) == prefix)
                atomicAdd(&sh.hist[(kk >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (warp == 0) {
            int s = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                s += (int)sh.hist[8 * lane + i];
            int incl = s;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off)
                    incl += y;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, incl >= k);
            const int src = hit ? __ffs(hit) - 1 : 31;
            if (lane == src) {
                int cum = incl - s, dsel = 8 * lane + 7;
                for (int i = 0; i < 8; ++i) {
                    const int h = (int)sh.hist[8 * lane + i];
                    if (cum + h >= k) {
                        dsel = 8 * lane + i;
                        break;
                    }
                    cum += h;
                }
                sh.bcast[0] = dsel;
                sh.bcast[1] = k - cum;
            }
        }
        __syncthreads();
        prefix |= (uint64_t)sh.bcast[0] << shift;
        mask |= (uint64_t)0xff << shift;
        k = sh.bcast[1];
        __syncthreads();
    }
    *rank_left = k;
    return prefix;
}

template <int KIND>
__global__ void __launch_bounds__(ETHREADS) k_evict(const EvictParams p)
{
    __shared__ Shared sh;
    const int unit = blockIdx.x, b = unit / p.Hkv, hk = unit % p.Hkv;
    int n = p.n[unit];
    if (n > p.C || n < 0) {
        if (threadIdx.x == 0)
            flag_error(p.status, DEV_CAPACITY);
        return;
    }
    if (KIND == EVICT_H2O && n < p.trigger)
        return;   // batched eviction: this unit has not reached its trigger
    const long T = p.seqlen[b];
    const int32_t *pos = p.pos + (size_t)unit * p.C;
    float *sc = p.scores ? p.scores + (size_t)unit * p.C : nullptr;

    // ---- 1. keep predicate
    uint64_t kth = 0;
    uint32_t pth = 0;
    int n_new = 0;
    if (KIND == EVICT_H2O) {
        const long rt = T - p.n_recent;
        auto is_recent = [&](int j) { return (long)pos[j] >= rt; };
        int n_rec = 0;
        for (int base = 0; base < n; base += ETHREADS) {
            const int j = base + threadIdx.x;
            n_rec += block_count(j < n && is_recent(j), sh);
        }
        const int n_cand = n - n_rec;
        const int take = min(p.n_heavy, n_cand);
        if (take >= n_cand)
            return; // nothing to drop
        n_new = n_rec + take;
        if (take > 0) {
            int left;
            kth = radix_select(
                n, take, 64,
                [&](int j) { return ((uint64_t)desc_bits(sc[j]) << 32) | (uint32_t)pos[j]; },
                [&](int j) { return !is_recent(j); }, &left, sh);
        }
    } else if (KIND == EVICT_STREAM) {
        int kept = 0;
        for (int base = 0; base < n; base += ETHREADS) {
            const int j = base + threadIdx.x;
            const bool k = j < n && ((long)pos[j] < p.n_sink || (long)pos[j] >= T - p.n_recent);
            kept += block_count(k, sh);
        }
        if (kept == n)
            return;
        n_new = kept;
    } else {
        int n_cand = 0;
        for (int base = 0; base < n; base += ETHREADS) {
            const int j = base + threadIdx.x;
            n_cand += block_count(j < n && pos[j] >= p.prompt_len, sh);
        }
        if (n_cand == 0)
            return;
        int n_keep = (int)((double)n_cand * p.keep_ratio);
        n_keep = n_keep < 1 ? 1 : (n_keep > n_cand ? n_cand : n_keep);
        if (n_keep == n_cand)
            return;
        n_new = n - n_cand + n_keep;
        auto rkey = [&](int j) {
            return philox_key(p.seed_lo, p.seed_hi, (uint32_t)pos[j], (uint32_t)hk, (uint32_t)b,
                              p.epoch);
        };
        int left;
        kth = radix_select(n, n_keep, 64, rkey, [&](int j) { return pos[j] >= p.prompt_len; },
                           &left, sh);
        // among candidates whose key equals the threshold keep the `left` lowest positions
        int left2;
        pth = (uint32_t)radix_select(
            n, left, 32, [&](int j) { return (uint64_t)(uint32_t)pos[j]; },
            [&](int j) { return pos[j] >= p.prompt_len && rkey(j) == kth; }, &left2, sh);
    }

    auto keep = [&](int j) -> bool {
        if (KIND == EVICT_H2O) {
            if ((long)pos[j] >= T - p.n_recent)
                return true;
            return (((uint64_t)desc_bits(sc[j]) << 32) | (uint32_t)pos[j]) <= kth &&
                   p.n_heavy > 0;
        } else if (KIND == EVICT_STREAM) {
            return (long)pos[j] < p.n_sink || (long)pos[j] >= T - p.n_recent;
        } else {
            if (pos[j] < p.prompt_len)
                return true;
            const uint64_t k = philox_key(p.seed_lo, p.seed_hi, (uint32_t)pos[j], (uint32_t)hk,
                                          (uint32_t)b, p.epoch);
            return k < kth || (k == kth && (uint32_t)pos[j] <= pth);
        }
    };

    // ---- 2. keep flags, taken once before any slot moves (moves change pos)
    for (int base = 0; base < n; base += ETHREADS) {
        const int j = base + threadIdx.x;
        const unsigned bits = __ballot_sync(0xffffffffu, j < n && keep(j));
        if ((threadIdx.x & 31) == 0 && j < n)
            sh.keep[j >> 5] = bits;
    }
    __syncthreads();
    auto kept = [&](int j) { return (sh.keep[j >> 5] >> (j & 31)) & 1u; };

    // ---- 3. compaction: k-th hole of [0, n_new) <- k-th kept slot of [n_new, n).
    // Holes and tail-kept slots are equal in number; ranks are assigned in
    // slot order in rounds of HOLE_CAP pairs.
    int n_pairs = 0;
    for (int base = 0; base < n_new; base += ETHREADS) {
        const int j = base + threadIdx.x;
        n_pairs += block_count(j < n_new && !kept(j), sh);
    }
    const int D = p.D;
    for (int round0 = 0; round0 < n_pairs; round0 += HOLE_CAP) {
        int seen = 0;
        for (int base = 0; base < n_new; base += ETHREADS) {
            const int j = base + threadIdx.x;
            const bool h = j < n_new && !kept(j);
            int tot;
            const int rk = seen + block_scan(h ? 1 : 0, &tot, sh);
            if (h && rk >= round0 && rk < round0 + HOLE_CAP)
                sh.hole[rk - round0] = j;
            seen += tot;
        }
        seen = 0;
        for (int base = n_new; base < n; base += ETHREADS) {
            const int j = base + threadIdx.x;
            const bool t = j < n && kept(j);
            int tot;
            const int rk = seen + block_scan(t ? 1 : 0, &tot, sh);
            if (t && rk >= round0 && rk < round0 + HOLE_CAP) {
                sh.mv_src[rk - round0] = j;
                sh.mv_dst[rk - round0] = sh.hole[rk - round0];
            }
            seen += tot;
        }
        __syncthreads();
        const int cnt = min(HOLE_CAP, n_pairs - round0);
        // move rows: one warp per pair; 16-byte chunks of K then V
        const int chunks = D / 8;
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        for (int k = warp; k < cnt; k += NWARPS) {
            const size_t src = (size_t)unit * p.C + sh.mv_src[k];
            const size_t dst = (size_t)unit * p.C + sh.mv_dst[k];
            const long rs = p.rows.row(unit, sh.mv_src[k]), rd = p.rows.row(unit, sh.mv_dst[k]);
            uint4 *K4 = reinterpret_cast<uint4 *>(p.K), *V4 = reinterpret_cast<uint4 *>(p.V);
            if (rs < 0 || rd < 0) {   // no page behind a slot: skip the row, flag it
                if (lane == 0)
                    flag_error(p.status, DEV_CAPACITY);
            } else {
                for (int ch = lane; ch < 2 * chunks; ch += 32) {
                    if (ch < chunks)
                        K4[rd * chunks + ch] = K4[rs * chunks + ch];
                    else
                        V4[rd * chunks + ch - chunks] = V4[rs * chunks + ch - chunks];
                }
            }
            if (lane == 0) {
                p.pos[dst] = p.pos[src];
                if (sc)
                    p.scores[dst] = p.scores[src];
            }
        }
        __syncthreads();
    }
    // freed slots start from a zero score when a later token is appended there
    if (sc)
        for (int j = n_new + threadIdx.x; j < n; j += ETHREADS)
            sc[j] = 0.f;
    if (threadIdx.x == 0)
        p.n[unit] = n_new;
}

// ------------------------------------------------------------------------
// Decode-sized caches (C <= WE_MAX_SLOTS): one warp per unit, warp-level
// primitives only (no CTA barriers), so every unit of the batch is resident at
// once.  Same keep rules and the same fill-the-holes-from-the-tail compaction.
// A second instance for C <= WE_SMALL_SLOTS (a 512-slot budget plus its decode
// slack) holds half the registers per lane, so four CTAs fit per SM instead of
// two and a 4096-unit batch runs in one round.
// ------------------------------------------------------------------------
constexpr int WE_WARPS = 8;
constexpr int WE_MAX_SLOTS = 1024;
constexpr int WE_SMALL_SLOTS = 576;

template <typename KeyFn, typename FiltFn>
__device__ uint64_t warp_radix_select(int n, int k, KeyFn key, FiltFn filt, uint32_t *hist)
{
    const int lane = threadIdx.x & 31;
    uint64_t prefix = 0, mask = 0;
    for (int shift = 56; shift >= 0; shift -= 8) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            hist[8 * lane + i] = 0;
        __syncwarp();
        for (int base = 0; base < n; base += 32) {
            const int j = base + lane;
            if (j < n && filt(j)) {
                const uint64_t kk = key(j);
                if ((kk & mask) == prefix)
                    atomicAdd(&hist[(kk >> shift) & 255u], 1u);
            }
        }
        __syncwarp();
        int s = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            s += (int)hist[8 * lane + i];
        int incl = s;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off)
                incl += y;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, incl >= k);
        const int src = hit ? __ffs(hit) - 1 : 31;
        int digit = 0, left = 0;
        if (lane == src) {
            int cum = incl - s;
            digit = 8 * lane + 7;
            for (int i = 0; i < 8; ++i) {
                const int h = (int)hist[8 * lane + i];
                if (cum + h >= k) {
                    digit = 8 * lane + i;
                    break;
                }
                cum += h;
            }
            left = k - cum;
        }
        digit = __shfl_sync(0xffffffffu, digit, src);
        k = __shfl_sync(0xffffffffu, left, src);
        prefix |= (uint64_t)digit << shift;
        mask |= (uint64_t)0xff << shift;
        __syncwarp();
    }
    return prefix;
}

template <int KIND, int MAXS>
__global__ void __launch_bounds__(WE_WARPS * 32, MAXS <= WE_SMALL_SLOTS ? 4 : 1)
    k_evict_warp(const EvictParams p, int n_units)
{
    static_assert(MAXS % 32 == 0, "whole words of slots");
    __shared__ uint32_t s_keep[WE_WARPS][MAXS / 32];
    __shared__ uint32_t s_hist[WE_WARPS][256];
    __shared__ uint16_t s_hole[WE_WARPS][MAXS / 2];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int unit = blockIdx.x * WE_WARPS + warp;
    if (unit >= n_units)
        return;
    const int n = p.n[unit];
    if (n > p.C || n < 0) {
        if (lane == 0)
            flag_error(p.status, DEV_CAPACITY);
        return;
    }
    if (KIND == EVICT_H2O && n < p.trigger)
        return;   // batched eviction: this unit has not reached its trigger
    const long T = p.seqlen[unit / p.Hkv];
    const int32_t *pos = p.pos + (size_t)unit * p.C;
    float *sc = p.scores ? p.scores + (size_t)unit * p.C : nullptr;
    uint32_t *keep = s_keep[warp];
    const long rt = T - p.n_recent;
    int n_new = 0;
    // the unit's positions (and H2O scores) in registers: slot 32 i + lane in element i,
    // every load issued before the first is used, so the scans below cost one round trip
    constexpr int NR = MAXS / 32;
    int32_t pr[NR];
    float sr[KIND == EVICT_H2O ? NR : 1];
#pragma unroll
    for (int i = 0; i < NR; ++i) {
        const int j = 32 * i + lane;
        pr[i] = j < n ? pos[j] : 0;
        if constexpr (KIND == EVICT_H2O)
            sr[i] = j < n ? sc[j] : 0.f;
    }

    if (KIND == EVICT_STREAM) {
#pragma unroll
        for (int i = 0; i < NR; ++i) {
            if (32 * i >= n)
                break;
            const int j = 32 * i + lane;
            const bool k = j < n && ((long)pr[i] < p.n_sink || (long)pr[i] >= rt);
            const unsigned m = __ballot_sync(0xffffffffu, k);
            if (lane == 0)
                keep[i] = m;
            n_new += __popc(m);
        }
        if (n_new == n)
            return;
    } else {
        int n_rec = 0;
#pragma unroll
        for (int i = 0; i < NR; ++i) {
            if (32 * i >= n)
                break;
            const int j = 32 * i + lane;
            const unsigned m = __ballot_sync(0xffffffffu, j < n && (long)pr[i] >= rt);
            if (lane == 0)
                keep[i] = m;
            n_rec += __popc(m);
        }
        const int take = min(p.n_heavy, n - n_rec);
        if (take >= n - n_rec)
            return;   // nothing to drop
        n_new = n_rec + take;
        auto key = [&](int j) { return ((uint64_t)desc_bits(sc[j]) << 32) | (uint32_t)pos[j]; };
        auto cand = [&](int j) { return (long)pos[j] < rt; };
        const int drops = n - n_rec - take;
        if (drops == 1) {
            // the decode step's case: the worst candidate -- the largest (descending
            // score, position) key -- leaves and the last slot moves into its place,
            // which is what the hole / tail compaction below does for a single hole
            uint64_t best = 0;
            int bj = -1;
#pragma unroll
            for (int i = 0; i < NR; ++i) {
                if (32 * i >= n)
                    break;
                const int j = 32 * i + lane;
                if (j < n && (long)pr[i] < rt) {
                    const uint64_t k = ((uint64_t)desc_bits(sr[i]) << 32) | (uint32_t)pr[i];
                    if (bj < 0 || k > best) {
                        best = k;
                        bj = j;
                    }
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const uint64_t ok = __shfl_xor_sync(0xffffffffu, best, off);
                const int oj = __shfl_xor_sync(0xffffffffu, bj, off);
                if (oj >= 0 && (bj < 0 || ok > best)) {
                    best = ok;
                    bj = oj;
                }
            }
            const int last = n - 1;
            if (bj != last) {
                const int chunks = p.D / 8;
                uint4 *K4 = reinterpret_cast<uint4 *>(p.K), *V4 = reinterpret_cast<uint4 *>(p.V);
                const long rs = p.rows.row(unit, last), rd = p.rows.row(unit, bj);
                if (rs < 0 || rd < 0) {   // no page behind a slot: skip the row, flag it
                    if (lane == 0)
                        flag_error(p.status, DEV_CAPACITY);
                } else {
                    for (int ch = lane; ch < 2 * chunks; ch += 32) {
                        if (ch < chunks)
                            K4[rd * chunks + ch] = K4[rs * chunks + ch];
                        else
                            V4[rd * chunks + ch - chunks] = V4[rs * chunks + ch - chunks];
                    }
                }
                if (lane == 0) {
                    p.pos[(size_t)unit * p.C + bj] = p.pos[(size_t)unit * p.C + last];
                    sc[bj] = sc[last];
                }
            }
            if (lane == 0) {
                sc[last] = 0.f;   // the freed slot starts from a zero score
                p.n[unit] = last;
            }
            return;
        }
        if (take > 0 && drops <= 4) {
            // few drops (the decode step drops one): keep every candidate, then remove
            // the worst -- the largest (descending score, position) key -- drops times
#pragma unroll
            for (int i = 0; i < NR; ++i) {
                if (32 * i >= n)
                    break;
                const int j = 32 * i + lane;
                const unsigned m = __ballot_sync(0xffffffffu, j < n && (long)pr[i] < rt);
                if (lane == 0)
                    keep[i] |= m;
            }
            __syncwarp();
            for (int d = 0; d < drops; ++d) {
                uint64_t best = 0;
                int bj = -1;
#pragma unroll
                for (int i = 0; i < NR; ++i) {
                    if (32 * i >= n)
                        break;
                    const int j = 32 * i + lane;
                    if (j < n && (long)pr[i] < rt && ((keep[i] >> lane) & 1u)) {
                        const uint64_t k = ((uint64_t)desc_bits(sr[i]) << 32) | (uint32_t)pr[i];
                        if (bj < 0 || k > best) {
                            best = k;
                            bj = j;
                        }
                    }
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    const uint64_t ok = __shfl_xor_sync(0xffffffffu, best, off);
                    const int oj = __shfl_xor_sync(0xffffffffu, bj, off);
                    if (oj >= 0 && (bj < 0 || ok > best)) {
                        best = ok;
                        bj = oj;
                    }
                }
                if (lane == 0)
                    keep[bj >> 5] &= ~(1u << (bj & 31));
                __syncwarp();
            }
        } else if (take > 0) {
            const uint64_t kth = warp_radix_select(n, take, key, cand, s_hist[warp]);
            for (int base = 0; base < n; base += 32) {
                const int j = base + lane;
                const unsigned m = __ballot_sync(0xffffffffu, j < n && cand(j) && key(j) <= kth);
                if (lane == 0)
                    keep[base >> 5] |= m;
            }
        }
    }
    __syncwarp();

    // holes of [0, n_new) by rank
    int nh = 0;
    for (int base = 0; base < n_new; base += 32) {
        const int j = base + lane;
        const bool h = j < n_new && !((keep[base >> 5] >> lane) & 1u);
        const unsigned m = __ballot_sync(0xffffffffu, h);
        if (h)
            s_hole[warp][nh + __popc(m & ((1u << lane) - 1u))] = (uint16_t)j;
        nh += __popc(m);
    }
    __syncwarp();
    // kept slots of [n_new, n) fill the holes in order; the warp moves one row at a time
    const int chunks = p.D / 8;
    uint4 *K4 = reinterpret_cast<uint4 *>(p.K), *V4 = reinterpret_cast<uint4 *>(p.V);
    int done = 0;
    for (int base = n_new; base < n; base += 32) {
        const int j = base + lane;
        const bool t = j < n && ((keep[j >> 5] >> (j & 31)) & 1u);
        unsigned m = __ballot_sync(0xffffffffu, t);
        while (m) {
            const int l = __ffs(m) - 1;
            m &= m - 1;
            const int hole = s_hole[warp][done++];
            const size_t src = (size_t)unit * p.C + base + l;
            const size_t dst = (size_t)unit * p.C + hole;
            const long rs = p.rows.row(unit, base + l), rd = p.rows.row(unit, hole);
            if (rs < 0 || rd < 0) {   // no page behind a slot: skip the row, flag it
                if (lane == 0)
                    flag_error(p.status, DEV_CAPACITY);
            } else {
                for (int ch = lane; ch < 2 * chunks; ch += 32) {
                    if (ch < chunks)
                        K4[rd * chunks + ch] = K4[rs * chunks + ch];
                    else
                        V4[rd * chunks + ch - chunks] = V4[rs * chunks + ch - chunks];
                }
            }
            if (lane == 0) {
                p.pos[dst] = p.pos[src];
                if (sc)
                    p.scores[dst] = p.scores[src];
            }
        }
    }
    // freed slots start from a zero score when a later token is appended there
    if (sc) {
        __syncwarp();
        for (int j = n_new + lane; j < n; j += 32)
            sc[j] = 0.f;
    }
    if (lane == 0)
        p.n[unit] = n_new;
}

// ------------------------------------------------------------------------
// Random eviction for caches of at most RF_MAX_SLOTS slots (the reasoning-trace
// cadence keeps ~2400 per unit): one 1024-thread CTA per unit with the unit's
// positions and Philox keys staged in shared memory, so every key is computed
// once.  The n_keep-th smallest (key, pos) is found with one 2048-bin histogram
// of the top 11 key bits: bins below the crossing bin are kept whole, bins above
// are dropped, and the few members of the crossing bin are ranked against each
// other exactly.  The compaction then moves all rows at once, a warp per row
// pair (16-byte chunks per lane) with eight pairs in flight per warp.
// ------------------------------------------------------------------------
constexpr int RF_THREADS = 1024;
constexpr int RF_WARPS = RF_THREADS / 32;
constexpr int RF_BINS = 2048;                 // top 11 key bits
constexpr int RF_SHIFT = 64 - 11;
constexpr int RF_MAX_SLOTS = 8192;            // u16 slot indices, one keep word per thread
constexpr int RF_UNROLL = 8;                  // moved rows in flight per warp

__host__ __device__ constexpr size_t rf_align(size_t x) { return (x + 15) & ~(size_t)15; }

constexpr int RF_MISC = 128;                  // ints: two scans' scratch, then scalars
constexpr int RF_SCAN_A = 0, RF_SCAN_B = 48, RF_SCALARS = 96;

// Shared-memory carve-up for capacity C (bytes); the layout below must match.
__host__ __device__ constexpr size_t rf_smem_bytes(int C)
{
    return rf_align((size_t)C * 8)                          // keys
           + rf_align((size_t)C * 4)                        // positions
           + rf_align((size_t)((C + 31) / 32) * 4)          // keep bitmask
           + rf_align((size_t)(C + 2) * 2)                  // bucket list / hole + tail lists
           + (size_t)RF_BINS * 4                            // histogram, then word lists
           + RF_MISC * 4;                                   // scan scratch + scalars
}

// Exclusive scan of one int per thread over the 1024-thread CTA; *total gets the
// sum.  `wsum` holds RF_WARPS + 1 ints that no other scan uses before the next
// barrier.  All threads must call it.
__device__ __forceinline__ int rf_scan(int v, int *total, int *wsum)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off)
            x += y;
    }
    if (lane == 31)
        wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        const int t = wsum[lane];
        int ti = t;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, ti, off);
            if (lane >= off)
                ti += y;
        }
        wsum[lane] = ti - t;         // exclusive prefix of warp totals
        if (lane == 31)
            wsum[RF_WARPS] = ti;     // grand total
    }
    __syncthreads();
    *total = wsum[RF_WARPS];
    return wsum[warp] + x - v;
}

__global__ void __launch_bounds__(RF_THREADS, 1) k_evict_random(const EvictParams p)
{
    extern __shared__ __align__(16) uint8_t rf_smem[];
    const int C = p.C;
    uint64_t *s_key = reinterpret_cast<uint64_t *>(rf_smem);
    int32_t *s_pos = reinterpret_cast<int32_t *>(rf_smem + rf_align((size_t)C * 8));
    uint32_t *s_keep = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(s_pos) +
                                                    rf_align((size_t)C * 4));
    const int nwords = (C + 31) / 32;
    uint16_t *s_list = reinterpret_cast<uint16_t *>(reinterpret_cast<uint8_t *>(s_keep) +
                                                    rf_align((size_t)nwords * 4));
    uint32_t *s_hist = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(s_list) +
                                                    rf_align((size_t)(C + 2) * 2));
    int *s_misc = reinterpret_cast<int *>(s_hist + RF_BINS);
    // [0] bucket list length, [1] bin, [2] keys below it, [3] bin size
    int *s_sc = s_misc + RF_SCALARS;

    const int unit = blockIdx.x, b = unit / p.Hkv, hk = unit % p.Hkv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t *pos = p.pos + (size_t)unit * C;
    const int n = p.n[unit];
    for (int i = tid; i < RF_BINS; i += RF_THREADS)
        s_hist[i] = 0;
    if (tid == 0)
        s_sc[0] = 0;
    __syncthreads();

    // ---- 1. positions and keys into shared memory, top-bit histogram of the candidates.
    // The position loads of a round do not wait for n (slots up to C are readable).
    constexpr int PU = 4;
    const int nv = n < C ? n : C;   // a count above C is flagged below, after the loads
    for (int base = 0; base < C; base += PU * RF_THREADS) {
        int32_t pv[PU];
#pragma unroll
        for (int u = 0; u < PU; ++u) {
            const int j = base + u * RF_THREADS + tid;
            pv[u] = j < C ? pos[j] : 0;
        }
#pragma unroll
        for (int u = 0; u < PU; ++u) {
            const int j = base + u * RF_THREADS + tid;
            if (j < nv) {
                s_pos[j] = pv[u];
                uint64_t k = ~0ull;
                if (pv[u] >= p.prompt_len) {
                    k = philox_key(p.seed_lo, p.seed_hi, (uint32_t)pv[u], (uint32_t)hk,
                                   (uint32_t)b, p.epoch);
                    atomicAdd(&s_hist[(uint32_t)(k >> RF_SHIFT)], 1u);
                }
                s_key[j] = k;
            }
        }
    }
    if (n > C || n < 0) {
        if (tid == 0)
            flag_error(p.status, DEV_CAPACITY);
        return;
    }
    __syncthreads();

    // ---- 2. candidate count (the histogram's total) and the bin holding the n_keep-th
    // smallest key, two bins per thread
    const int h0 = (int)s_hist[2 * tid], h1 = (int)s_hist[2 * tid + 1];
    int n_cand;
    const int ex = rf_scan(h0 + h1, &n_cand, s_misc + RF_SCAN_A);
    if (n_cand == 0)
        return;
    int n_keep = (int)((double)n_cand * p.keep_ratio);
    n_keep = n_keep < 1 ? 1 : (n_keep > n_cand ? n_cand : n_keep);
    if (n_keep == n_cand)
        return;
    const int n_new = n - n_cand + n_keep;
    if (ex < n_keep && n_keep <= ex + h0 + h1) {
        const bool first = n_keep <= ex + h0;
        s_sc[1] = first ? 2 * tid : 2 * tid + 1;
        s_sc[2] = first ? ex : ex + h0;
        s_sc[3] = first ? h0 : h1;
    }
    __syncthreads();
    const uint32_t bstar = (uint32_t)s_sc[1];
    const int need = n_keep - s_sc[2];   // members of bin bstar to keep, in [1, s_sc[3]]
    const bool whole = need == s_sc[3];  // the whole bin is kept (the usual case)

    // ---- 3. keep flags: every prompt slot and the candidates of lower bins (of bin bstar
    // too when it is kept whole); otherwise bin bstar's members go to a list and are
    // decided by their exact rank among themselves
    for (int base = 0; base < n; base += RF_THREADS) {
        const int j = base + tid;
        bool kp = false;
        if (j < n) {
            if (s_pos[j] < p.prompt_len) {
                kp = true;
            } else {
                const uint32_t bin = (uint32_t)(s_key[j] >> RF_SHIFT);
                kp = bin < bstar || (whole && bin == bstar);
                if (!whole && bin == bstar)
                    s_list[atomicAdd(&s_sc[0], 1)] = (uint16_t)j;
            }
        }
        const unsigned m = __ballot_sync(0xffffffffu, kp);
        if (lane == 0 && base + 32 * warp < n)
            s_keep[(base >> 5) + warp] = m;
    }
    __syncthreads();
    if (!whole) {
        const int m_b = s_sc[0];
        for (int t = tid; t < m_b; t += RF_THREADS) {
            const int j = s_list[t];
            const uint64_t kj = s_key[j];
            const int32_t pj = s_pos[j];
            int rank = 0;
            for (int i = 0; i < m_b; ++i) {
                const int o = s_list[i];
                const uint64_t ko = s_key[o];
                rank += (ko < kj || (ko == kj && s_pos[o] < pj)) ? 1 : 0;
            }
            if (rank < need)
                atomicOr(&s_keep[j >> 5], 1u << (j & 31));
        }
        __syncthreads();
    }

    // ---- 4. hole and tail lists (k-th hole of [0, n_new) <- k-th kept slot of [n_new, n)):
    // per 32-slot word its hole and tail bits and their ranks (one thread per word), then
    // one warp per word writes the slots at their ranks
    uint16_t *s_hole = s_list;                       // ranks [0, pairs)
    uint16_t *s_tail = s_list + (C + 2) / 2;         // pairs <= min(n_new, n - n_new) <= C / 2
    uint32_t *s_hw = s_hist, *s_tw = s_hist + 256;   // nwords <= 256
    int *s_wb = reinterpret_cast<int *>(s_hist + 512);
    const int wn = (n + 31) / 32;
    int n_pairs;
    {
        uint32_t hb = 0, tb = 0;
        if (tid < wn) {
            const uint32_t w = s_keep[tid];
            const int lo = 32 * tid;
            const uint32_t valid = (n - lo >= 32) ? 0xffffffffu : ((1u << (n - lo)) - 1u);
            const uint32_t below = (n_new - lo >= 32) ? 0xffffffffu
                                   : (n_new - lo <= 0) ? 0u : ((1u << (n_new - lo)) - 1u);
            hb = ~w & below & valid;
            tb = w & ~below & valid;
        }
        // hole counts in the low 16 bits, tail counts in the high 16 (totals <= 8192)
        int both;
        const int exw = rf_scan(__popc(hb) | (__popc(tb) << 16), &both, s_misc + RF_SCAN_B);
        n_pairs = both & 0xffff;
        if (tid < wn) {
            s_hw[tid] = hb;
            s_tw[tid] = tb;
            s_wb[tid] = exw;
        }
    }
    __syncthreads();
    for (int wd = warp; wd < wn; wd += RF_WARPS) {
        const uint32_t hb = s_hw[wd], tb = s_tw[wd];
        const int wb = s_wb[wd];
        const uint32_t lt = (1u << lane) - 1u;
        if ((hb >> lane) & 1u)
            s_hole[(wb & 0xffff) + __popc(hb & lt)] = (uint16_t)(32 * wd + lane);
        if ((tb >> lane) & 1u)
            s_tail[(wb >> 16) + __popc(tb & lt)] = (uint16_t)(32 * wd + lane);
    }
    __syncthreads();

    // ---- 5. moves: a warp (half a warp at D = 64) per pair, lane c copies 16-byte chunk c
    // of the pair's K row then V row; RF_UNROLL pairs per warp in flight
    const int chunks = p.D / 8;                  // per row
    const int per_pair = 2 * chunks;             // 32 (D = 128) or 16 (D = 64)
    const int ppw = 32 / per_pair;
    const int c = lane % per_pair;
    const bool isv = c >= chunks;
    const int cc = isv ? c - chunks : c;
    uint4 *base4 = reinterpret_cast<uint4 *>(isv ? p.V : p.K);
    int32_t *gpos = p.pos + (size_t)unit * C;
    for (int k0 = 0; k0 < n_pairs; k0 += RF_WARPS * ppw * RF_UNROLL) {
        uint4 v[RF_UNROLL];
        int rd[RF_UNROLL];
#pragma unroll
        for (int u = 0; u < RF_UNROLL; ++u) {
            const int k = k0 + (u * RF_WARPS + warp) * ppw + lane / per_pair;
            rd[u] = -1;
            if (k < n_pairs) {
                const int src = s_tail[k], dst = s_hole[k];
                const long rs = p.rows.row(unit, src), rdl = p.rows.row(unit, dst);
                if (rs < 0 || rdl < 0) {   // no page behind a slot: skip the row, flag it
                    if (c == 0)
                        flag_error(p.status, DEV_CAPACITY);
                } else {
                    v[u] = base4[(size_t)rs * chunks + cc];
                    rd[u] = (int)rdl;
                }
                if (c == 0)
                    gpos[dst] = s_pos[src];
            }
        }
#pragma unroll
        for (int u = 0; u < RF_UNROLL; ++u)
            if (rd[u] >= 0)
                base4[(size_t)rd[u] * chunks + cc] = v[u];
    }
    if (tid == 0)
        p.n[unit] = n_new;
}

} // namespace

cudaError_t launch_evict(const EvictLaunch &e, cudaStream_t s)
{
    EvictParams p{};
    p.Hkv = e.c.Hkv;
    p.D = e.c.D;
    p.C = e.c.C;
    p.K = e.c.K;
    p.V = e.c.V;
    p.pos = e.c.pos;
    p.n = e.c.n;
    p.seqlen = e.c.seqlen;
    p.scores = e.scores;
    p.n_heavy = e.n_heavy;
    p.n_recent = e.n_recent;
    p.n_sink = e.n_sink;
    p.prompt_len = e.prompt_len;
    p.trigger = e.trigger;
    p.rows = SlotRows{e.c.block_table, e.c.C, e.c.num_pages};
    p.keep_ratio = e.keep_ratio;
    p.seed_lo = (uint32_t)(e.seed & 0xffffffffu);
    p.seed_hi = (uint32_t)(e.seed >> 32);
    p.epoch = e.epoch;
    p.status = dev_status_ptr();
    const int units = e.c.B * e.c.Hkv;
    const bool small = e.c.C <= WE_MAX_SLOTS;
    const int wgrid = (units + WE_WARPS - 1) / WE_WARPS;
    switch (e.kind) {
    case EVICT_H2O:
        if (e.c.C <= WE_SMALL_SLOTS)
            k_evict_warp<EVICT_H2O, WE_SMALL_SLOTS><<<wgrid, WE_WARPS * 32, 0, s>>>(p, units);
        else if (small)
            k_evict_warp<EVICT_H2O, WE_MAX_SLOTS><<<wgrid, WE_WARPS * 32, 0, s>>>(p, units);
        else
            k_evict<EVICT_H2O><<<units, ETHREADS, 0, s>>>(p);
        break;
    case EVICT_STREAM:
        if (e.c.C <= WE_SMALL_SLOTS)
            k_evict_warp<EVICT_STREAM, WE_SMALL_SLOTS><<<wgrid, WE_WARPS * 32, 0, s>>>(p, units);
        else if (small)
            k_evict_warp<EVICT_STREAM, WE_MAX_SLOTS><<<wgrid, WE_WARPS * 32, 0, s>>>(p, units);
        else
            k_evict<EVICT_STREAM><<<units, ETHREADS, 0, s>>>(p);
        break;
    default:
        if (e.c.C <= RF_MAX_SLOTS) {
            const int smem = (int)rf_smem_bytes(e.c.C);
            const cudaError_t err = set_smem_once(reinterpret_cast<const void *>(k_evict_random),
                                                  (int)rf_smem_bytes(RF_MAX_SLOTS));
            if (err != cudaSuccess)
                return err;
            k_evict_random<<<units, RF_THREADS, smem, s>>>(p);
        } else {
            k_evict<EVICT_RANDOM><<<units, ETHREADS, 0, s>>>(p);
        }
        break;
    }
    return cudaGetLastError();
}

} // namespace kvc
