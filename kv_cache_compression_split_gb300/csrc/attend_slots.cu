// attend_slots.cu -- split-KV decode attention over an fp16 slot cache, plus
// the split combine (shared with the KIVI kernel).
//
// One CTA handles one (sequence b, KV head hk, split) work item: the g query
// heads of hk against the split's token range.  A producer warp streams K and
// V tiles of 64 tokens into shared memory with 2-D TMA (128-byte swizzle,
// mbarrier-tracked, NSTAGE deep); four consumer warps each take 16 tokens of a
// tile and compute, with mma.sync m16n8k16 (tokens on M, query heads on N):
//   S^T = K_tile Q^T          (16 tokens x 8 heads, fp32)
//   online softmax per head   (running max m, running sum l, base-2 exponent)
//   O^T += V_tile^T P^T       (D x 8 heads, fp32; P^T is the S^T fragment
//                              transposed in registers with movmatrix)
// The four warps' (m, l, O) are merged through shared memory at the end.
// With one split the CTA writes o and lse directly.  With several splits each
// CTA writes its partial (m, l, unnormalised O) to a workspace that the combine
// kernel merges -- except for the fused H2O score update with 2..8 splits: then
// the splits of a unit form one thread-block cluster, each CTA leaves its
// partial in its shared memory, and after a cluster barrier the CTAs read each
// other's partials through distributed shared memory, write o and lse, and
// fold their own tokens' probabilities (logits still on chip) into the scores,
// all in one launch.
//
// Method: scaled dot-product attention of one decode query over the kept
// cache ("Rethinking KV Cache Compression" guide, §16 "Prefill、decode、TP 的
// 性能账": each decode step reads the whole kept history, so the step is
// bandwidth bound and every byte is read once).
#include "kvc_device.cuh"
#include "kvc_internal.h"

#include <math.h>

namespace kvc {

namespace {

constexpr int NCW = 4;                 // consumer warps (16 tokens of a tile each)
constexpr int NTHREADS = (NCW + 1) * 32;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

// Where the fused H2O launch keeps the unit's logits instead of an output array:
//   LM_SMEM  in shared memory ([8][LSM_SLOTS] fp32), with fewer stages to make room;
//   LM_REGS  in the registers of the thread that computed them (up to LREG_TILES
//            tiles, i.e. C <= 576 slots), which leaves all stages in place.
constexpr int LM_NONE = 0, LM_SMEM = 1, LM_REGS = 2;
constexpr int LSM_SLOTS = H2O_ONCHIP_MAX_SLOTS;
constexpr int LREG_TILES = 9;
template <int D, int LMODE = LM_NONE> struct SlotCfg {
    static constexpr bool LSM = LMODE == LM_SMEM;
    static constexpr int NBOX = D / 64;                 // 64-half (128-byte) boxes per row
    static constexpr int TILE_BYTES = TILE * D * 2;     // one K or V tile
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;  // K + V
    static constexpr int NSTAGE = LSM ? ((D == 128) ? 2 : 4) : ((D == 128) ? 3 : 6);
    static constexpr int LSM_BYTES = LSM ? 8 * LSM_SLOTS * 4 : 0;
    // the mbarriers (full, empty, new token), then the decode step's new K and V rows
    static constexpr int BAR_BYTES = (2 * NSTAGE + 1) * 8;
    static constexpr int NEWTOK_OFF = (BAR_BYTES + 15) / 16 * 16;
    // then the H2O step's copy of the unit's positions (up to LSM_SLOTS)
    static constexpr int SPOS_OFF = NEWTOK_OFF + 2 * D * 2;
    static constexpr int SMEM = NSTAGE * STAGE_BYTES + LSM_BYTES + 1024 + SPOS_OFF + LSM_SLOTS * 4;
    static_assert(NCW * (8 * D + 16) * 4 <= NSTAGE * STAGE_BYTES, "combine scratch must fit");
    // this CTA's merged partial for the cluster merge, after the warps' scratch
    static constexpr int CP_OFF = NCW * (8 * D + 16) * 4;
    static_assert(CP_OFF + (8 * D + 16) * 4 <= NSTAGE * STAGE_BYTES, "cluster partial must fit");
};
constexpr int MAX_CLUSTER = 8;   // portable thread-block cluster size

struct SlotParams {
    int Hq, Hkv, C, g;
    int splits, tiles_per_split;
    const uint16_t *q;
    uint16_t *o;
    const int32_t *n;               // valid slots per unit
    float *logits, *lse;
    float *part_o, *part_ml;
    float scale, scale_log2;
    int cluster;                    // > 1: the splits of a unit are one cluster, merged on chip
    float *h2o_scores;              // optional: add this step's probabilities (fused update)
    float h2o_keep, h2o_add;        // scores = keep * scores + add * p
    SlotRows rows;                  // dense or paged K / V rows
    int *status;
    // fused decode steps (STEP_H2O / STEP_STREAM): the new token of every unit, the cache
    // arrays the step writes, and the method's window
    const uint16_t *k_new, *v_new;  // [B, Hkv, 1, D]
    uint16_t *K, *V;
    int32_t *pos, *n_w, *seqlen;
    int n_heavy, n_recent, n_sink;
};

// Decode-step modes of the slot kernel: plain attention, or one whole decode step of a
// method in one launch (append + attention + the method's eviction).
constexpr int STEP_NONE = 0, STEP_H2O = 1, STEP_STREAM = 2;

__device__ __forceinline__ void consumer_bar()
{
    asm volatile("bar.sync 1, %0;" ::"n"(NCW * 32) : "memory");
}

// Slots [0, n) of each unit are valid.
//
// STEP_H2O / STEP_STREAM (one split): the unit's new token, at position P = seqlen[b],
// joins the attention from k_new / v_new (the cache is not written until the end), and
// the step then writes exactly one K/V row:
//   H2O     the scores are updated as in the fused accumulate, the new token gets its
//           own; if the unit held n_heavy + n_recent slots, the worst non-recent slot by
//           (score desc, position asc) is the one dropped, and the new token takes its
//           slot (with its score); otherwise the token goes to slot n and n grows.
//   STREAM  the token that left the window with the previous step (position
//           P - n_recent - 1, when >= n_sink) is not attended and gives up its slot;
//           otherwise the token goes to slot n.
// seqlen[b] advances once all Hkv CTAs of sequence b have read it: each adds 1 << 24 on
// arrival, and the last to arrive removes the counts and adds 1.
template <int D, int LMODE, int STEP>
__global__ void __launch_bounds__(NTHREADS, 2)
    k_attend_slots(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const SlotParams p)
{
    using Cfg = SlotCfg<D, LMODE>;
    constexpr bool LSM = Cfg::LSM, LREG = LMODE == LM_REGS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_align1024(smem_raw);
    float *lsm = reinterpret_cast<float *>(smem + Cfg::NSTAGE * Cfg::STAGE_BYTES);  // LSM only
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cfg::NSTAGE * Cfg::STAGE_BYTES +
                                                  Cfg::LSM_BYTES);
    uint64_t *empty = full + Cfg::NSTAGE;
    uint64_t *ntbar = empty + Cfg::NSTAGE;   // the decode step's new K/V rows have landed
    uint8_t *newtok = reinterpret_cast<uint8_t *>(full) + Cfg::NEWTOK_OFF;   // K row, V row
    const int32_t *spos = reinterpret_cast<const int32_t *>(reinterpret_cast<uint8_t *>(full) +
                                                            Cfg::SPOS_OFF);   // H2O step

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int unit = blockIdx.x / p.splits, split = blockIdx.x % p.splits;
    const int b = unit / p.Hkv, hk = unit % p.Hkv;

    // token range of this split
    int n_valid = p.n[unit];
    const bool n_bad = n_valid > p.C || n_valid < 0;   // flagged; a decode step then writes nothing
    if (n_valid > p.C) {
        if (threadIdx.x == 0)
            flag_error(p.status, DEV_CAPACITY);
        n_valid = p.C;
    }
    if (n_valid < 0)
        n_valid = 0;
    const int t_begin = split * p.tiles_per_split * TILE;
    const int t_end = min(n_valid, t_begin + p.tiles_per_split * TILE);
    const int ntiles = t_end > t_begin ? (t_end - t_begin + TILE - 1) / TILE : 0;

    __shared__ int s_step[4];   // [0] P, [1] the stream step's leaving slot, [2] H2O victim
    if (threadIdx.x == 0) {
        for (int i = 0; i < Cfg::NSTAGE; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], NCW);
        }
        // decode steps: complete when the new rows have landed (the producer's bulk copies)
        // and the position P has been read (consumer warp 1)
        mbar_init(ntbar, STEP != STEP_NONE ? 2 : 1);
        fence_mbar_init();
        s_step[1] = -1;
        s_step[2] = -1;
    }
    __syncthreads();

    if (warp == NCW) {
        // ---------------- producer: the step's new K/V rows (bulk copies), then TMA K/V
        // tiles into the stage ring
        if (STEP != STEP_NONE && lane == 0) {
            // the H2O step also copies the unit's positions (C is a multiple of 4, so the
            // row starts on 16 bytes; n_valid rounded up to 4 slots stays within C)
            const int pbytes = STEP == STEP_H2O ? (n_valid + 3) / 4 * 16 : 0;
            mbar_arrive_expect_tx(ntbar, 2 * D * 2 + pbytes);
            bulk_load(newtok, p.k_new + (size_t)unit * D, D * 2, ntbar);
            bulk_load(newtok + D * 2, p.v_new + (size_t)unit * D, D * 2, ntbar);
            if (pbytes > 0)
                bulk_load(reinterpret_cast<uint8_t *>(full) + Cfg::SPOS_OFF,
                          p.pos + (size_t)unit * p.C, pbytes, ntbar);
        }
        if (lane == 0 && ntiles > 0) {
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            for (int i = 0; i < ntiles; ++i) {
                // a tile is one page in the paged layout (t_begin is a multiple of 64);
                // a bad table entry reads past the pool (zero fill) and is flagged
                long row = p.rows.row(unit, t_begin + i * TILE);
                if (row < 0) {
                    flag_error(p.status, DEV_CAPACITY);
                    row = (long)p.rows.num_pages * TILE;
                }
                const int st = i % Cfg::NSTAGE;
                if (i >= Cfg::NSTAGE && !mbar_wait(&empty[st], ((i / Cfg::NSTAGE) & 1) ^ 1)) {
                    flag_error(p.status, DEV_TIMEOUT);
                    break;
                }
                uint8_t *kt = smem + st * Cfg::STAGE_BYTES;
                uint8_t *vt = kt + Cfg::TILE_BYTES;
                mbar_arrive_expect_tx(&full[st], Cfg::STAGE_BYTES);
#pragma unroll
                for (int j = 0; j < Cfg::NBOX; ++j) {
                    tma_load_2d(kt + j * TILE * 128, &tmK, &full[st], 64 * j, (int)row);
                    tma_load_2d(vt + j * TILE * 128, &tmV, &full[st], 64 * j, (int)row);
                }
            }
        }
        __syncwarp();
        if (p.cluster > 1) {   // the consumers' two cluster barriers
            cluster_sync_all();
            cluster_sync_all();
        }
        return;
    }

    // ---------------- consumers
    const int r = lane >> 2, c = lane & 3;
    const int mi = lane >> 3, ri = lane & 7;

    if (STEP != STEP_NONE && warp == 1 && lane == 0) {
        // the new token's position: every CTA of the sequence adds an arrival and the last
        // one advances seqlen.  The round trip overlaps the first tiles' loads; the threads
        // that need P wait on ntbar.
        const int old = atomicAdd(&p.seqlen[b], 1 << 24);
        if ((old >> 24) + 1 == p.Hkv)
            atomicAdd(&p.seqlen[b], 1 - (p.Hkv << 24));
        s_step[0] = old & 0xffffff;
        mbar_arrive(ntbar);
    }

    // Q^T as the B operand: b0 = Q[head r][16s + 2c, +1], b1 = Q[head r][16s + 2c + 8, +1]
    uint32_t qf[D / 16][2];
    {
        const bool hv = r < p.g;
        const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
            p.q + ((size_t)b * p.Hq + hk * p.g + (hv ? r : 0)) * D);
#pragma unroll
        for (int s = 0; s < D / 16; ++s) {
            qf[s][0] = hv ? qrow[8 * s + c] : 0u;
            qf[s][1] = hv ? qrow[8 * s + c + 4] : 0u;
        }
    }

    if constexpr (STEP == STEP_STREAM) {
        // the slot of the token that left the window with the previous step (P first)
        if (!mbar_wait(ntbar, 0))
            flag_error(p.status, DEV_TIMEOUT);
        const long leave = (long)s_step[0] - p.n_recent - 1;
        if (leave >= p.n_sink) {
            const int32_t *up = p.pos + (size_t)unit * p.C;
            for (int j = threadIdx.x; j < n_valid; j += NCW * 32)
                if ((long)up[j] == leave)
                    s_step[1] = j;
        }
        consumer_bar();
    }
    const int skip = STEP == STEP_STREAM ? s_step[1] : -1;   // a slot not attended

    float acc[D / 16][4];
#pragma unroll
    for (int m = 0; m < D / 16; ++m)
        acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.f;
    float m_run0 = -INFINITY, m_run1 = -INFINITY, l_run0 = 0.f, l_run1 = 0.f;
    const int h0 = 2 * c, h1 = 2 * c + 1;
    float *lg0 = nullptr, *lg1 = nullptr;
    const int lofs = LSM ? t_begin : 0;   // the shared-memory logits hold this split's tokens
    if (LSM) {
        lg0 = h0 < p.g ? lsm + h0 * LSM_SLOTS : nullptr;
        lg1 = h1 < p.g ? lsm + h1 * LSM_SLOTS : nullptr;
    } else if (p.logits) {
        const size_t rowbase = ((size_t)b * p.Hq + hk * p.g) * p.C;
        lg0 = h0 < p.g ? p.logits + rowbase + (size_t)h0 * p.C : nullptr;
        lg1 = h1 < p.g ? p.logits + rowbase + (size_t)h1 * p.C : nullptr;
    }

    // one tile: wait for it, fold it into the running state, hand the stage back;
    // lr receives this thread's four logits (tokens r, r + 8 of the warp's 16 x
    // heads 2c, 2c + 1), the values the other storage modes write
    auto do_tile = [&](int i, float (&lr)[4]) -> bool {
        const int st = i % Cfg::NSTAGE;
        lr[0] = lr[1] = lr[2] = lr[3] = -INFINITY;
        if (!mbar_wait(&full[st], (i / Cfg::NSTAGE) & 1)) {
            flag_error(p.status, DEV_TIMEOUT);
            return false;
        }
        const int tok0 = t_begin + i * TILE + 16 * warp;
        if (tok0 < t_end) {
            const uint32_t kbase = smem_u32(smem + st * Cfg::STAGE_BYTES);
            const uint32_t vbase = kbase + Cfg::TILE_BYTES;

            float sa[4] = {0.f, 0.f, 0.f, 0.f};
            const int krow = 16 * warp + ri + 8 * (mi & 1);
#pragma unroll
            for (int s = 0; s < D / 16; ++s) {
                const int ch = 2 * s + (mi >> 1);
                uint32_t a0, a1, a2, a3;
                ldsm_x4(swz128(kbase + (ch >> 3) * TILE * 128, krow, ch & 7), a0, a1, a2, a3);
                mma16816(sa, a0, a1, a2, a3, qf[s][0], qf[s][1]);
            }

            const int ta = tok0 + r, tb = tok0 + r + 8;
            const bool va = ta < t_end && ta != skip, vb = tb < t_end && tb != skip;
            if (lg0) {
                if (va) lg0[ta - lofs] = sa[0] * p.scale;
                if (vb) lg0[tb - lofs] = sa[2] * p.scale;
            }
            if (lg1) {
                if (va) lg1[ta - lofs] = sa[1] * p.scale;
                if (vb) lg1[tb - lofs] = sa[3] * p.scale;
            }
            const float x0 = va ? sa[0] * p.scale_log2 : -INFINITY;
            const float x1 = va ? sa[1] * p.scale_log2 : -INFINITY;
            const float x2 = vb ? sa[2] * p.scale_log2 : -INFINITY;
            const float x3 = vb ? sa[3] * p.scale_log2 : -INFINITY;
            lr[0] = sa[0] * p.scale;
            lr[1] = sa[1] * p.scale;
            lr[2] = sa[2] * p.scale;
            lr[3] = sa[3] * p.scale;
            float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            const float mn0 = fmaxf(m_run0, mx0), mn1 = fmaxf(m_run1, mx1);
            const float al0 = mn0 == -INFINITY ? 1.f : ex2(m_run0 - mn0);
            const float al1 = mn1 == -INFINITY ? 1.f : ex2(m_run1 - mn1);
            const float p0 = mn0 == -INFINITY ? 0.f : ex2(x0 - mn0);
            const float p2 = mn0 == -INFINITY ? 0.f : ex2(x2 - mn0);
            const float p1 = mn1 == -INFINITY ? 0.f : ex2(x1 - mn1);
            const float p3 = mn1 == -INFINITY ? 0.f : ex2(x3 - mn1);
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
            const uint32_t pb0 = movmatrix_t(pack_half2(p0, p1));
            const uint32_t pb1 = movmatrix_t(pack_half2(p2, p3));
            const int vrow = 16 * warp + ri + 8 * (mi >> 1);
#pragma unroll
            for (int m = 0; m < D / 16; ++m) {
                const int ch = 2 * m + (mi & 1);
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(swz128(vbase + (ch >> 3) * TILE * 128, vrow, ch & 7), a0, a1, a2, a3);
                mma16816(acc[m], a0, a1, a2, a3, pb0, pb1);
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(&empty[st]);
        return true;
    };
    float lreg[LREG ? LREG_TILES : 1][4];   // LM_REGS: every tile's scores of this thread
    // LM_REGS: lane c == 0 of each quad loads the old scores of its tokens now, so the
    // loads are in flight while the tiles stream instead of at the end
    float old[LREG ? LREG_TILES : 1][2];
    if constexpr (LREG) {
#pragma unroll
        for (int i = 0; i < LREG_TILES; ++i) {
            const int ta = t_begin + i * TILE + 16 * warp + r, tb = ta + 8;
            const float *sc = p.h2o_scores + (size_t)unit * p.C;
            const bool upd = p.h2o_scores && p.part_o == nullptr && c == 0 && i < ntiles;
            old[i][0] = upd && ta < t_end ? sc[ta] : 0.f;
            old[i][1] = upd && tb < t_end ? sc[tb] : 0.f;
        }
    }
    if constexpr (LREG) {
#pragma unroll
        for (int i = 0; i < LREG_TILES; ++i) {
            lreg[i][0] = lreg[i][1] = lreg[i][2] = lreg[i][3] = -INFINITY;
            if (i < ntiles && !do_tile(i, lreg[i]))
                break;
        }
    } else {
        for (int i = 0; i < ntiles; ++i)
            if (!do_tile(i, lreg[0]))
                break;
    }

    // ---------------- decode steps: the new token joins warp 0's running state (row 0 of
    // a 16-row block; the padding rows have no mass)
    float lnew[2] = {-INFINITY, -INFINITY};   // warp 0, lanes 0-3: its logits, heads 2c, 2c + 1
    if constexpr (STEP != STEP_NONE) {
        if (warp == 0) {
            // K for S^T = K Q^T: lanes 0-3 (row 0) take words 8s + c and 8s + c + 4 of the
            // new K row; V for O^T += V^T P^T: lanes with c == 0 (token column 0) take
            // channels 16m + r and 16m + r + 8 of the new V row
            if (!mbar_wait(ntbar, 0))
                flag_error(p.status, DEV_TIMEOUT);
            const uint32_t *k32 = reinterpret_cast<const uint32_t *>(newtok);
            const uint16_t *v16 = reinterpret_cast<const uint16_t *>(newtok + D * 2);
            float sa[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int s = 0; s < D / 16; ++s)
                mma16816(sa, r == 0 ? k32[8 * s + c] : 0u, 0u, r == 0 ? k32[8 * s + c + 4] : 0u,
                         0u, qf[s][0], qf[s][1]);
            const bool va = r == 0;
            if (va) {
                lnew[0] = sa[0] * p.scale;
                lnew[1] = sa[1] * p.scale;
            }
            const float x0 = va ? sa[0] * p.scale_log2 : -INFINITY;
            const float x1 = va ? sa[1] * p.scale_log2 : -INFINITY;
            float mx0 = x0, mx1 = x1;
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            const float mn0 = fmaxf(m_run0, mx0), mn1 = fmaxf(m_run1, mx1);
            const float al0 = mn0 == -INFINITY ? 1.f : ex2(m_run0 - mn0);
            const float al1 = mn1 == -INFINITY ? 1.f : ex2(m_run1 - mn1);
            const float p0 = mn0 == -INFINITY ? 0.f : ex2(x0 - mn0);
            const float p1 = mn1 == -INFINITY ? 0.f : ex2(x1 - mn1);
            m_run0 = mn0;
            m_run1 = mn1;
            l_run0 = l_run0 * al0 + p0;
            l_run1 = l_run1 * al1 + p1;
#pragma unroll
            for (int m = 0; m < D / 16; ++m) {
                acc[m][0] *= al0;
                acc[m][1] *= al1;
                acc[m][2] *= al0;
                acc[m][3] *= al1;
            }
            const uint32_t pb0 = movmatrix_t(pack_half2(p0, p1));
#pragma unroll
            for (int m = 0; m < D / 16; ++m)
                mma16816(acc[m], c == 0 ? (uint32_t)v16[16 * m + r] : 0u,
                         c == 0 ? (uint32_t)v16[16 * m + r + 8] : 0u, 0u, 0u, pb0, 0u);
        }
    }

    // ---------------- merge the four warps
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l_run0 += __shfl_xor_sync(0xffffffffu, l_run0, off);
        l_run1 += __shfl_xor_sync(0xffffffffu, l_run1, off);
    }
    consumer_bar();   // every consumer is past its last shared-memory read
    float *redO = reinterpret_cast<float *>(smem);        // [NCW][8][D]
    float *redM = redO + NCW * 8 * D;                     // [NCW][8]
    float *redL = redM + NCW * 8;                         // [NCW][8]
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
    const bool clustered = p.cluster > 1;
    const bool single = !clustered && p.part_o == nullptr;
    float *cp_o = reinterpret_cast<float *>(smem + Cfg::CP_OFF);   // [8][D] cluster partial
    float *cp_ml = cp_o + 8 * D;                                    // [8][2] max (log2), sum
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
        if (clustered) {
            cp_o[h * D + d] = os;
            if (d == 0) {
                cp_ml[2 * h] = ls > 0.f ? ms : -INFINITY;
                cp_ml[2 * h + 1] = ls;
            }
        } else if (single) {
            const size_t oi = ((size_t)b * p.Hq + hk * p.g + h) * D + d;
            p.o[oi] = __half_as_ushort(__float2half_rn(ls > 0.f ? os / ls : 0.f));
            if (d == 0 && p.lse)
                p.lse[(size_t)b * p.Hq + hk * p.g + h] =
                    ls > 0.f ? (ms + __log2f(ls)) * LN2 : -INFINITY;
        } else {
            const size_t pi = ((size_t)unit * p.splits + split) * p.g + h;
            p.part_o[pi * D + d] = os;
            if (d == 0) {
                p.part_ml[2 * pi] = ls > 0.f ? ms : -INFINITY;
                p.part_ml[2 * pi + 1] = ls;
            }
        }
    }
    __shared__ float s_lse2[8];   // log2-domain lse per head (H2O epilogue)
    if (clustered) {
        // merge the cluster's partials: split s has weight 2^(m_s - M) in head h
        __shared__ float s_w[8][MAX_CLUSTER], s_l[8];
        __syncwarp();
        cluster_sync_all();   // every CTA's partial is written and visible
        if (threadIdx.x < p.g) {
            const int h = threadIdx.x;
            float mm = -INFINITY;
            for (int r = 0; r < p.cluster; ++r)
                mm = fmaxf(mm, ld_cluster_f32(cp_ml + 2 * h, r));
            float ls = 0.f;
            for (int r = 0; r < p.cluster; ++r) {
                const float m = ld_cluster_f32(cp_ml + 2 * h, r);
                const float w = m == -INFINITY ? 0.f : ex2(m - mm);
                s_w[h][r] = w;
                ls += w * ld_cluster_f32(cp_ml + 2 * h + 1, r);
            }
            s_l[h] = ls;
            s_lse2[h] = ls > 0.f ? mm + __log2f(ls) : INFINITY;
            if (split == 0 && p.lse)
                p.lse[(size_t)b * p.Hq + hk * p.g + h] =
                    ls > 0.f ? (mm + __log2f(ls)) * LN2 : -INFINITY;
        }
        consumer_bar();
        for (int e = split * NCW * 32 + threadIdx.x; e < p.g * D; e += p.cluster * NCW * 32) {
            const int h = e / D, d = e % D;
            float os = 0.f;
            for (int r = 0; r < p.cluster; ++r)
                if (s_w[h][r] != 0.f)
                    os += s_w[h][r] * ld_cluster_f32(cp_o + h * D + d, r);
            const size_t oi = ((size_t)b * p.Hq + hk * p.g + h) * D + d;
            p.o[oi] = __half_as_ushort(__float2half_rn(s_l[h] > 0.f ? os / s_l[h] : 0.f));
        }
        __syncwarp();
        cluster_sync_all();   // no CTA leaves while another still reads its partial
    }
    // H2O decode step: the worst non-recent slot by (score desc, position asc), tracked as
    // the largest key (descending-score bits << 32 | position) while the scores are written
    long h2o_rt = 0;   // recent: positions >= rt (set once P is known)
    unsigned long long vkey = 0ull;
    int vslot = -1;
    auto candidate = [&](int slot, int32_t ps, float score) {
        if constexpr (STEP == STEP_H2O) {
            if ((long)ps < h2o_rt) {
                const unsigned long long k =
                    ((unsigned long long)desc_bits(score) << 32) | (uint32_t)ps;
                if (vslot < 0 || k > vkey) {
                    vkey = k;
                    vslot = slot;
                }
            }
        }
    };
    float s_new = 0.f;   // H2O step: the new token's score (warp 0, lane 0)
    if ((single || clustered) && p.h2o_scores) {
        // H2O decode scores: score[j] += sum_h exp(logit_hj - lse_h) over this unit's
        // query heads, for this CTA's tokens (logits kept by this CTA; log2 domain here)
        if (!clustered && threadIdx.x < p.g) {
            const int h = threadIdx.x;
            float ms = -INFINITY;
#pragma unroll
            for (int w = 0; w < NCW; ++w)
                ms = fmaxf(ms, redM[w * 8 + h]);
            float ls = 0.f;
#pragma unroll
            for (int w = 0; w < NCW; ++w) {
                const float mw = redM[w * 8 + h];
                ls += (mw == -INFINITY ? 0.f : ex2(mw - ms)) * redL[w * 8 + h];
            }
            s_lse2[h] = ls > 0.f ? ms + __log2f(ls) : INFINITY;
        }
        consumer_bar();
        float *sc = p.h2o_scores + (size_t)unit * p.C;
        if constexpr (STEP == STEP_H2O) {
            // the positions copied at the start and P (their phase completed long ago)
            if (!mbar_wait(ntbar, 0))
                flag_error(p.status, DEV_TIMEOUT);
            h2o_rt = (long)s_step[0] + 1 - p.n_recent;
            // the new token's probabilities (warp 0, lanes 0-3 hold heads 2c, 2c + 1), added
            // in head order like every other slot's
            if (warp == 0) {
                const float L0 = h0 < p.g ? s_lse2[h0] : 0.f, L1 = h1 < p.g ? s_lse2[h1] : 0.f;
                const float e0 = h0 < p.g ? ex2(fmaf(lnew[0], LOG2E, -L0)) : 0.f;
                const float e1 = h1 < p.g ? ex2(fmaf(lnew[1], LOG2E, -L1)) : 0.f;
                float add = 0.f;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    add += __shfl_sync(0xffffffffu, e0, q);
                    add += __shfl_sync(0xffffffffu, e1, q);
                }
                s_new = fmaf(0.f, p.h2o_keep, add * p.h2o_add);
            }
        }
        if constexpr (LREG) {
            // the same arithmetic as the other storage modes: lane c == 0 of each quad
            // gathers the probabilities of heads 0 .. 7 for tokens r and r + 8 of every
            // tile (heads 2c, 2c + 1 come from lane c) and adds them in head order
            const float L0 = h0 < p.g ? s_lse2[h0] : 0.f, L1 = h1 < p.g ? s_lse2[h1] : 0.f;
#pragma unroll
            for (int i = 0; i < LREG_TILES; ++i) {
                if (i >= ntiles)
                    break;
                const float e[4] = {h0 < p.g ? ex2(fmaf(lreg[i][0], LOG2E, -L0)) : 0.f,
                                    h1 < p.g ? ex2(fmaf(lreg[i][1], LOG2E, -L1)) : 0.f,
                                    h0 < p.g ? ex2(fmaf(lreg[i][2], LOG2E, -L0)) : 0.f,
                                    h1 < p.g ? ex2(fmaf(lreg[i][3], LOG2E, -L1)) : 0.f};
                float add_a = 0.f, add_b = 0.f;
#pragma unroll
                for (int q = 0; q < 4; ++q) {   // heads 2q, 2q + 1 from lane 4r + q
                    const int src = (lane & ~3) + q;
                    add_a += __shfl_sync(0xffffffffu, e[0], src);
                    add_a += __shfl_sync(0xffffffffu, e[1], src);
                    add_b += __shfl_sync(0xffffffffu, e[2], src);
                    add_b += __shfl_sync(0xffffffffu, e[3], src);
                }
                const int ta = t_begin + i * TILE + 16 * warp + r, tb = ta + 8;
                if (c == 0 && ta < t_end) {
                    const float v = fmaf(old[i][0], p.h2o_keep, add_a * p.h2o_add);
                    sc[ta] = v;
                    if constexpr (STEP == STEP_H2O)
                        candidate(ta, spos[ta], v);
                }
                if (c == 0 && tb < t_end) {
                    const float v = fmaf(old[i][1], p.h2o_keep, add_b * p.h2o_add);
                    sc[tb] = v;
                    if constexpr (STEP == STEP_H2O)
                        candidate(tb, spos[tb], v);
                }
            }
        } else {
            const float *lrow = LSM ? lsm : p.logits + ((size_t)b * p.Hq + hk * p.g) * p.C;
            const size_t lstride = LSM ? LSM_SLOTS : p.C;
            // four slots per thread per round, every load issued before any is used
            constexpr int U = 4;
            for (int j0 = t_begin + threadIdx.x; j0 < t_end; j0 += U * NCW * 32) {
                float add[U], old[U];
                int32_t ps[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int j = j0 + u * NCW * 32;
                    add[u] = 0.f;
                    old[u] = j < t_end ? sc[j] : 0.f;
                    ps[u] = STEP == STEP_H2O && j < t_end ? spos[j] : 0;
                }
                // all heads' logits of the round in flight at once (g <= 8)
                float lg[8][U];
#pragma unroll
                for (int h = 0; h < 8; ++h)
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int j = j0 + u * NCW * 32;
                        lg[h][u] =
                            h < p.g && j < t_end ? lrow[(size_t)h * lstride + (j - lofs)] : 0.f;
                    }
#pragma unroll
                for (int h = 0; h < 8; ++h)
                    if (h < p.g)
#pragma unroll
                        for (int u = 0; u < U; ++u)
                            add[u] += ex2(fmaf(lg[h][u], LOG2E, -s_lse2[h]));
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int j = j0 + u * NCW * 32;
                    if (j < t_end) {
                        const float v = fmaf(old[u], p.h2o_keep, add[u] * p.h2o_add);
                        sc[j] = v;
                        candidate(j, ps[u], v);
                    }
                }
            }
        }
    }

    // ---------------- decode steps: the one row the step writes
    if constexpr (STEP != STEP_NONE) {
        __shared__ unsigned long long s_vkey[NCW];
        __shared__ int s_vslot[NCW];
        if constexpr (STEP == STEP_H2O) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const unsigned long long ok = __shfl_xor_sync(0xffffffffu, vkey, off);
                const int os = __shfl_xor_sync(0xffffffffu, vslot, off);
                if (os >= 0 && (vslot < 0 || ok > vkey)) {
                    vkey = ok;
                    vslot = os;
                }
            }
            if (lane == 0) {
                s_vkey[warp] = vkey;
                s_vslot[warp] = vslot;
            }
            consumer_bar();
        }
        if (warp == 0) {
            const int P = s_step[0];
            int slot = -1;
            bool grow = false;
            if constexpr (STEP == STEP_H2O) {
                const int budget = p.n_heavy + p.n_recent;
                if (n_valid < budget) {
                    slot = n_valid;
                    grow = true;
                } else {
                    // at budget: the worst candidate leaves and the new token takes its slot
                    unsigned long long best = 0ull;
#pragma unroll
                    for (int w = 0; w < NCW; ++w)
                        if (s_vslot[w] >= 0 && (slot < 0 || s_vkey[w] > best)) {
                            best = s_vkey[w];
                            slot = s_vslot[w];
                        }
                    if (h2o_rt > (long)P) {
                        // no recent window: the new token is a candidate too, and may be the
                        // one that leaves (then nothing is written)
                        const unsigned long long knew =
                            ((unsigned long long)desc_bits(s_new) << 32) | (uint32_t)P;
                        if (slot < 0 || knew > best)
                            slot = -2;
                    }
                    if (n_valid > budget)
                        slot = -1;   // more than one slot would have to go: not a decode step
                }
            } else {
                slot = skip >= 0 ? skip : n_valid;
                grow = skip < 0;
            }
            if (grow && slot >= p.C)
                slot = -1;
            if (slot == -2) {
                // the new token left at once: the cache keeps its slots
            } else if (slot < 0 || n_bad || P >= (1 << 24) - 1) {
                if (lane == 0)
                    flag_error(p.status, DEV_CAPACITY);
            } else {
                const long row = p.rows.row(unit, slot);
                constexpr int CH = D / 8;   // 16-byte chunks per row
                if (row < 0) {
                    if (lane == 0)
                        flag_error(p.status, DEV_CAPACITY);
                } else if (lane < 2 * CH) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(newtok) + lane;
                    uint4 *dst = reinterpret_cast<uint4 *>(lane < CH ? p.K : p.V) +
                                 (size_t)row * CH + (lane % CH);
                    *dst = *src;
                }
                if (lane == 0) {
                    p.pos[(size_t)unit * p.C + slot] = P;
                    if constexpr (STEP == STEP_H2O)
                        p.h2o_scores[(size_t)unit * p.C + slot] = s_new;
                    if (grow)
                        p.n_w[unit] = n_valid + 1;
                }
            }
        }
    }
}

// Merge split partials: o = sum_s 2^(m_s - m*) O_s / sum_s 2^(m_s - m*) l_s.
// One warp per (sequence, query head) row, eight rows per block: the lanes read
// the splits' (m, l) pairs 32 at a time, then every lane walks the splits for
// its D/32 channels, so the partial rows stream in with 16-byte loads.
constexpr int COMBINE_ROWS = 8;

template <int D>
__global__ void __launch_bounds__(32 * COMBINE_ROWS)
    k_combine(int rows, int unit0, int Hq, int Hkv, int g, int splits,
              const float *__restrict__ part_o, const float *__restrict__ part_ml,
              uint16_t *__restrict__ o, float *__restrict__ lse)
{
    constexpr int V = D / 32;   // channels per lane
    static_assert(V == 2 || V == 4, "head dim 64 or 128");
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * COMBINE_ROWS + (threadIdx.x >> 5);
    if (row >= rows)
        return;
    // row = (unit - unit0) * g + h; the unit is (b, hk), its query heads hk g .. hk g + g-1
    const int j = row / g, h = row % g, unit = unit0 + j;
    const int bh = (unit / Hkv) * Hq + (unit % Hkv) * g + h;
    const size_t base = ((size_t)j * splits) * g + h;
    const float *ml = part_ml + 2 * base;   // split sp at ml[2 sp g], ml[2 sp g + 1]
    float ms = -INFINITY;
    for (int sp = lane; sp < splits; sp += 32)
        ms = fmaxf(ms, ml[2 * (size_t)sp * g]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        ms = fmaxf(ms, __shfl_xor_sync(0xffffffffu, ms, off));
    float ls = 0.f;
    for (int sp = lane; sp < splits; sp += 32) {
        const float m = ml[2 * (size_t)sp * g];
        ls += (m == -INFINITY ? 0.f : ex2(m - ms)) * ml[2 * (size_t)sp * g + 1];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        ls += __shfl_xor_sync(0xffffffffu, ls, off);
    float os[V];
#pragma unroll
    for (int v = 0; v < V; ++v)
        os[v] = 0.f;
#pragma unroll 4
    for (int sp = 0; sp < splits; ++sp) {
        const float m = ml[2 * (size_t)sp * g];
        const float w = m == -INFINITY ? 0.f : ex2(m - ms);
        const float *src = part_o + (base + (size_t)sp * g) * D + V * lane;
        if constexpr (V == 4) {
            const float4 x = *reinterpret_cast<const float4 *>(src);
            os[0] = fmaf(w, x.x, os[0]);
            os[1] = fmaf(w, x.y, os[1]);
            os[2] = fmaf(w, x.z, os[2]);
            os[3] = fmaf(w, x.w, os[3]);
        } else {
            const float2 x = *reinterpret_cast<const float2 *>(src);
            os[0] = fmaf(w, x.x, os[0]);
            os[1] = fmaf(w, x.y, os[1]);
        }
    }
    uint32_t packed[V / 2];
#pragma unroll
    for (int v = 0; v < V / 2; ++v) {
        const float lo = ls > 0.f ? os[2 * v] / ls : 0.f, hi = ls > 0.f ? os[2 * v + 1] / ls : 0.f;
        packed[v] = (uint32_t)__half_as_ushort(__float2half_rn(lo)) |
                    ((uint32_t)__half_as_ushort(__float2half_rn(hi)) << 16);
    }
    uint16_t *dst = o + (size_t)bh * D + V * lane;
    if constexpr (V == 4)
        *reinterpret_cast<uint2 *>(dst) = make_uint2(packed[0], packed[1]);
    else
        *reinterpret_cast<uint32_t *>(dst) = packed[0];
    if (lane == 0 && lse)
        lse[bh] = ls > 0.f ? (ms + __log2f(ls)) * LN2 : -INFINITY;
}

template <int D, int LMODE, int STEP = STEP_NONE>
cudaError_t launch_slots_impl(const CUtensorMap &tk, const CUtensorMap &tv, const SlotParams &sp,
                              int grid, cudaStream_t s)
{
    using Cfg = SlotCfg<D, LMODE>;
    const cudaError_t e =
        set_smem_once(reinterpret_cast<const void *>(k_attend_slots<D, LMODE, STEP>), Cfg::SMEM);
    if (e != cudaSuccess)
        return e;
    if (sp.cluster <= 1) {
        k_attend_slots<D, LMODE, STEP><<<grid, NTHREADS, Cfg::SMEM, s>>>(tk, tv, sp);
        return cudaGetLastError();
    }
    // the splits of a unit (consecutive blocks) form one cluster
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = Cfg::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = sp.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_attend_slots<D, LMODE, STEP>, tk, tv, sp);
}

} // namespace

cudaError_t launch_attend_slots(const AttendLaunch &a, cudaStream_t s)
{
    const int units = a.B * a.Hkv;
    CUtensorMap tk, tv;
    const uint64_t rows =
        a.block_table ? (uint64_t)a.num_pages * TILE : (uint64_t)units * a.C;
    if (!encode_tmap_2d_f16(&tk, a.K, a.D, rows, 64, TILE) ||
        !encode_tmap_2d_f16(&tv, a.V, a.D, rows, 64, TILE))
        return cudaErrorInvalidValue;
    SlotParams sp{};
    sp.Hq = a.Hq;
    sp.Hkv = a.Hkv;
    sp.C = a.C;
    sp.g = a.Hq / a.Hkv;
    sp.splits = a.splits;
    sp.tiles_per_split = a.tiles_per_split;
    sp.q = a.q;
    sp.o = a.o;
    sp.n = a.n;
    // one split, or 2..8 splits merged in their cluster: o, lse and the fused H2O update in
    // this launch; more splits: partials to the workspace, merged by the combine kernel
    const bool on_chip = a.splits == 1 || a.cluster;
    if (a.cluster && (a.splits < 2 || a.splits > MAX_CLUSTER))
        return cudaErrorInvalidValue;
    sp.logits = a.logits;
    sp.lse = on_chip ? a.lse : nullptr;
    sp.part_o = on_chip ? nullptr : a.part_o;
    sp.part_ml = on_chip ? nullptr : a.part_ml;
    sp.scale = a.scale;
    sp.scale_log2 = a.scale * LOG2E;
    sp.cluster = a.cluster ? a.splits : 1;
    sp.h2o_scores = on_chip ? a.h2o_scores : nullptr;
    sp.h2o_keep = a.h2o_keep;
    sp.h2o_add = a.h2o_add;
    sp.rows = SlotRows{a.block_table, a.C, a.num_pages};
    sp.status = dev_status_ptr();
    const int grid = units * a.splits;
    // fused H2O without a logits array: each CTA keeps its split's logits on chip (in
    // registers up to LREG_TILES tiles, else in shared memory, at most LSM_SLOTS; checked
    // by the caller)
    const bool lsm = a.h2o_scores && !a.logits;
    if (lsm && (!on_chip || a.tiles_per_split * TILE > LSM_SLOTS))
        return cudaErrorInvalidValue;
    const int lmode = !lsm ? LM_NONE : (a.tiles_per_split <= LREG_TILES ? LM_REGS : LM_SMEM);
    cudaError_t e;
    if (a.D == 128)
        e = lmode == LM_REGS   ? launch_slots_impl<128, LM_REGS>(tk, tv, sp, grid, s)
            : lmode == LM_SMEM ? launch_slots_impl<128, LM_SMEM>(tk, tv, sp, grid, s)
                               : launch_slots_impl<128, LM_NONE>(tk, tv, sp, grid, s);
    else
        e = lmode == LM_REGS   ? launch_slots_impl<64, LM_REGS>(tk, tv, sp, grid, s)
            : lmode == LM_SMEM ? launch_slots_impl<64, LM_SMEM>(tk, tv, sp, grid, s)
                               : launch_slots_impl<64, LM_NONE>(tk, tv, sp, grid, s);
    if (e != cudaSuccess || on_chip)
        return e;
    return launch_combine(a.B, a.Hq, a.Hkv, a.D, a.splits, 0, a.B * a.Hkv, a.part_o, a.part_ml,
                          a.o, a.lse, s);
}

cudaError_t launch_decode_step(const StepLaunch &a, cudaStream_t s)
{
    const kvc_slot_cache &c = a.c;
    const int units = c.B * c.Hkv;
    CUtensorMap tk, tv;
    const uint64_t rows = c.block_table ? (uint64_t)c.num_pages * TILE : (uint64_t)units * c.C;
    if (!encode_tmap_2d_f16(&tk, c.K, c.D, rows, 64, TILE) ||
        !encode_tmap_2d_f16(&tv, c.V, c.D, rows, 64, TILE))
        return cudaErrorInvalidValue;
    const bool h2o = a.scores != nullptr;
    if (h2o && c.C > LSM_SLOTS)
        return cudaErrorInvalidValue;
    SlotParams sp{};
    sp.Hq = a.Hq;
    sp.Hkv = c.Hkv;
    sp.C = c.C;
    sp.g = a.Hq / c.Hkv;
    sp.splits = 1;
    sp.tiles_per_split = (c.C + TILE - 1) / TILE;
    sp.q = a.q;
    sp.o = a.o;
    sp.n = c.n;
    sp.lse = a.lse;
    sp.scale = a.scale;
    sp.scale_log2 = a.scale * LOG2E;
    sp.cluster = 1;
    sp.h2o_scores = a.scores;
    sp.h2o_keep = a.h2o_keep;
    sp.h2o_add = a.h2o_add;
    sp.rows = SlotRows{c.block_table, c.C, c.num_pages};
    sp.status = dev_status_ptr();
    sp.k_new = a.k_new;
    sp.v_new = a.v_new;
    sp.K = c.K;
    sp.V = c.V;
    sp.pos = c.pos;
    sp.n_w = c.n;
    sp.seqlen = c.seqlen;
    sp.n_heavy = a.n_heavy;
    sp.n_recent = a.n_recent;
    sp.n_sink = a.n_sink;
    if (!h2o)
        return c.D == 128 ? launch_slots_impl<128, LM_NONE, STEP_STREAM>(tk, tv, sp, units, s)
                          : launch_slots_impl<64, LM_NONE, STEP_STREAM>(tk, tv, sp, units, s);
    const bool regs = c.C <= LREG_TILES * TILE;
    if (c.D == 128)
        return regs ? launch_slots_impl<128, LM_REGS, STEP_H2O>(tk, tv, sp, units, s)
                    : launch_slots_impl<128, LM_SMEM, STEP_H2O>(tk, tv, sp, units, s);
    return regs ? launch_slots_impl<64, LM_REGS, STEP_H2O>(tk, tv, sp, units, s)
                : launch_slots_impl<64, LM_SMEM, STEP_H2O>(tk, tv, sp, units, s);
}

cudaError_t launch_combine(int B, int Hq, int Hkv, int D, int splits, int unit0, int n_units,
                           const float *part_o, const float *part_ml, uint16_t *o, float *lse,
                           cudaStream_t s)
{
    (void)B;
    const int g = Hq / Hkv;
    const int rows = n_units * g;
    if (rows <= 0)
        return cudaSuccess;
    const int grid = (rows + COMBINE_ROWS - 1) / COMBINE_ROWS;
    if (D == 128)
        k_combine<128><<<grid, 32 * COMBINE_ROWS, 0, s>>>(rows, unit0, Hq, Hkv, g, splits, part_o,
                                                          part_ml, o, lse);
    else
        k_combine<64><<<grid, 32 * COMBINE_ROWS, 0, s>>>(rows, unit0, Hq, Hkv, g, splits, part_o,
                                                         part_ml, o, lse);
    return cudaGetLastError();
}

} // namespace kvc
