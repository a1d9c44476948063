// api.cu -- the extern "C" entry points of libkvc.so: argument validation,
// launch planning, tensor-map encoding and the device status word.
// Every entry point validates on the host and enqueues nothing on error.
#include "kvc_internal.h"

#include <cudaTypedefs.h>
#include <limits.h>
#include <math.h>
#include <mutex>
#include <vector>

namespace kvc {

namespace {

__device__ int g_status;   // KVC_DEV_* bits, one word per device

constexpr int MAX_DEVICES = 64;
constexpr int EVICT_MAX_SLOTS = 65536;

int *g_status_ptr[MAX_DEVICES];
int g_sm_count[MAX_DEVICES];
std::mutex g_mu;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

int current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES)
        return -1;
    return dev;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool head_dim_ok(int D) { return D == 64 || D == 128; }

} // namespace

int *dev_status_ptr()
{
    const int dev = current_device();
    if (dev < 0)
        return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess)
            return nullptr;
        g_status_ptr[dev] = static_cast<int *>(p);
    }
    return g_status_ptr[dev];
}

int sm_count()
{
    const int dev = current_device();
    if (dev < 0)
        return 1;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_sm_count[dev]) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        g_sm_count[dev] = v > 0 ? v : 1;
    }
    return g_sm_count[dev];
}

namespace {
struct KernelDeviceEntry {
    const void *func;
    int dev;
    int value;   // resident CTAs (resident_ctas) or 1 (set_smem_once)
    bool occupancy;
};
std::vector<KernelDeviceEntry> g_kernel_entries;   // guarded by g_mu
} // namespace

cudaError_t set_smem_once(const void *func, int bytes)
{
    const int dev = current_device();
    if (dev < 0)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    for (const KernelDeviceEntry &e : g_kernel_entries)
        if (e.func == func && e.dev == dev && !e.occupancy)
            return cudaSuccess;
    const cudaError_t err =
        cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (err == cudaSuccess)
        g_kernel_entries.push_back({func, dev, 1, false});
    return err;
}

int resident_ctas(const void *func, int threads, int smem)
{
    const int dev = current_device();
    if (dev < 0)
        return 1;
    const int sms = sm_count();
    std::lock_guard<std::mutex> lk(g_mu);
    for (const KernelDeviceEntry &e : g_kernel_entries)
        if (e.func == func && e.dev == dev && e.occupancy)
            return e.value;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, func, threads, smem) != cudaSuccess)
        per_sm = 1;
    const int v = (per_sm > 0 ? per_sm : 1) * sms;
    g_kernel_entries.push_back({func, dev, v, true});
    return v;
}

bool encode_tmap_2d_f16(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                        uint32_t box_inner, uint32_t box_rows)
{
    auto fn = encode_fn();
    if (!fn || !aligned16(base) || rows == 0 || rows > (uint64_t)INT_MAX)
        return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

SlotAttendPlan plan_attend(int units, int tiles_per_unit, int requested, int max_splits)
{
    SlotAttendPlan pl{1, tiles_per_unit > 0 ? tiles_per_unit : 1};
    if (tiles_per_unit <= 0)
        return pl;
    int S = 1;
    if (requested > 0) {
        S = requested < tiles_per_unit ? requested : tiles_per_unit;
    } else {
        // Cost in tile-times (one SM streaming one tile at its share of HBM bandwidth):
        // the whole cache at the full-chip rate, or the busiest SM's CTAs one after another
        // (one CTA already draws about an SM's share), plus ~1.5 per round of two resident
        // CTAs per SM for a CTA's start and merge, plus 2 for merging split partials.
        // Measured on the LLaMA-7B, reasoning-trace and heavy-load shapes: 128 or more
        // units run fastest unsplit; a few long units need splits to fill the SMs.
        const double sms = (double)sm_count();
        double best = 1e300;
        int smax = tiles_per_unit < 64 ? tiles_per_unit : 64;
        if (smax > max_splits)
            smax = max_splits > 0 ? max_splits : 1;
        for (int s = 1; s <= smax; ++s) {
            const double ctas = (double)units * s;
            const double per_cta = ceil(tiles_per_unit / (double)s);
            const double stream = fmax((double)units * tiles_per_unit / sms, ceil(ctas / sms) * per_cta);
            const double cost = stream + 1.5 * ceil(ctas / (2.0 * sms)) + (s > 1 ? 2.0 : 0.0);
            if (cost < best - 1e-9) {
                best = cost;
                S = s;
            }
        }
    }
    pl.splits = S;
    pl.tiles_per_split = (tiles_per_unit + S - 1) / S;
    pl.splits = (tiles_per_unit + pl.tiles_per_split - 1) / pl.tiles_per_split;
    return pl;
}

namespace {

kvc_status check_slot_cache(const kvc_slot_cache *c)
{
    if (!c || !c->K || !c->V || !c->pos || !c->n || !c->seqlen)
        return KVC_ERR_INVALID_ARG;
    if (c->B <= 0 || c->Hkv <= 0 || c->C <= 0)
        return KVC_ERR_INVALID_ARG;
    if (!head_dim_ok(c->D))
        return KVC_ERR_UNSUPPORTED;
    if (!aligned16(c->K) || !aligned16(c->V) || !aligned16(c->pos))
        return KVC_ERR_INVALID_ARG;
    if ((long long)c->B * c->Hkv * c->C > (long long)INT_MAX)
        return KVC_ERR_UNSUPPORTED;
    if (c->block_table) {   // paged layout: whole pages per unit, a pool of num_pages
        if (c->C % KVC_PAGE_SLOTS != 0 || c->num_pages <= 0)
            return KVC_ERR_INVALID_ARG;
        if ((long long)c->num_pages * KVC_PAGE_SLOTS > (long long)INT_MAX)
            return KVC_ERR_UNSUPPORTED;
    }
    return KVC_OK;
}

kvc_status check_quant_cache(const kvc_quant_cache *c)
{
    if (!c || !c->k_blocks || !c->v_blocks || !c->k_res || !c->v_res || !c->len)
        return KVC_ERR_INVALID_ARG;
    if (c->B <= 0 || c->Hkv <= 0 || c->R < 0 || c->Cq < 0 || c->Cq % KIVI_G != 0)
        return KVC_ERR_INVALID_ARG;
    if (!head_dim_ok(c->D) || (c->bits != 2 && c->bits != 4))
        return KVC_ERR_UNSUPPORTED;
    if (c->block_table) {   // paged layout: whole pages of 4 groups, a pool of num_pages
        if (c->Cq % (KVC_KIVI_GROUP * KVC_KIVI_PAGE_GROUPS) != 0 || c->num_pages <= 0)
            return KVC_ERR_INVALID_ARG;
    }
    if (!c->k_gear != !c->v_gear)
        return KVC_ERR_INVALID_ARG;
    if (c->k_gear) {        // GEAR side blocks
        if (!aligned16(c->k_gear) || !aligned16(c->v_gear))
            return KVC_ERR_INVALID_ARG;
    }
    if (!aligned16(c->k_blocks) || !aligned16(c->v_blocks) || !aligned16(c->k_res) ||
        !aligned16(c->v_res))
        return KVC_ERR_INVALID_ARG;
    if ((long long)c->B * c->Hkv * (c->R + KIVI_G) > (long long)INT_MAX)
        return KVC_ERR_UNSUPPORTED;
    return KVC_OK;
}

kvc_status from_cuda(cudaError_t e) { return e == cudaSuccess ? KVC_OK : KVC_ERR_CUDA; }

struct AttendPlanFull {
    kvc_status st;
    int B, Hkv, D;
    SlotAttendPlan plan;
    int full_units;  // KIVI with plan.splits > 1: units 0 .. full_units-1 run unsplit
    bool cluster;   // slot caches: 2..8 splits merged in a thread-block cluster
    size_t ws;
};

AttendPlanFull plan_full(const kvc_attend_args *a)
{
    AttendPlanFull f{};
    f.st = KVC_ERR_INVALID_ARG;
    if (!a)
        return f;
    if (a->kind == KVC_KIND_SLOTS) {
        if (check_slot_cache(a->slots) != KVC_OK) {
            f.st = check_slot_cache(a->slots);
            return f;
        }
        f.B = a->slots->B;
        f.Hkv = a->slots->Hkv;
        f.D = a->slots->D;
        const int tiles = (a->slots->C + TILE - 1) / TILE;
        const int splits = a->num_splits;
        if (splits < 0)
            return f;
        if (a->h2o_scores && !a->logits) {
            // fused H2O with the logits on chip: every split keeps at most
            // H2O_ONCHIP_MAX_SLOTS logits and the splits merge in one cluster
            const int tmax = H2O_ONCHIP_MAX_SLOTS / TILE;
            const int need = (tiles + tmax - 1) / tmax;
            if (splits > SLOT_CLUSTER_MAX)
                return f;
            if (need > SLOT_CLUSTER_MAX || (splits > 0 && (tiles + splits - 1) / splits > tmax)) {
                f.st = KVC_ERR_UNSUPPORTED;
                return f;
            }
            f.plan = plan_attend(f.B * f.Hkv, tiles, splits, SLOT_CLUSTER_MAX);
            if (f.plan.tiles_per_split > tmax)
                f.plan = plan_attend(f.B * f.Hkv, tiles, need);
        } else {
            f.plan = plan_attend(f.B * f.Hkv, tiles, splits);
        }
        // the fused H2O update merges its splits inside their cluster (the logits stay with
        // the CTA that computed them); plain attention merges through the workspace, which
        // measured as fast or faster for 2-4 splits of small batches
        f.cluster = a->h2o_scores && f.plan.splits > 1 && f.plan.splits <= SLOT_CLUSTER_MAX;
        f.ws = f.plan.splits > 1 && !f.cluster
                   ? (size_t)f.B * a->Hq * f.plan.splits * (f.D + 2) * sizeof(float)
                   : 0;
    } else if (a->kind == KVC_KIND_KIVI) {
        if (check_quant_cache(a->quant) != KVC_OK) {
            f.st = check_quant_cache(a->quant);
            return f;
        }
        f.B = a->quant->B;
        f.Hkv = a->quant->Hkv;
        f.D = a->quant->D;
        // quantised tiles of four groups; the residual ring joins the last split
        const int tiles = (a->quant->Cq / KIVI_G + 3) / 4;
        const int units = f.B * f.Hkv;
        f.plan = plan_attend(units, tiles > 0 ? tiles : 1, a->num_splits);
        f.full_units = 0;
        if (a->num_splits <= 0 && f.plan.splits == 1 && tiles >= 2) {
            // The persistent CTAs (three per SM, two for GEAR) take whole units in
            // rounds.  When the last round fills at most half of them, only its units
            // are split (up to four ways), so that every CTA ends with about the same
            // work; the other units still run whole, without partials.
            const int ctas = (a->quant->k_gear ? 2 : 3) * sm_count();
            const int tail = ctas > 0 ? units % ctas : 0;
            if (units > ctas && tail > 0 && 2 * tail <= ctas) {
                int st = ctas / tail;
                st = st < 4 ? st : 4;
                st = st < tiles ? st : tiles;
                const int per = (tiles + st - 1) / st;
                f.plan.splits = (tiles + per - 1) / per;
                f.plan.tiles_per_split = per;
                f.full_units = f.plan.splits > 1 ? units - tail : 0;
            }
        }
        const int split_units = units - f.full_units;
        f.ws = f.plan.splits > 1 ? (size_t)split_units * (a->Hq / f.Hkv) * f.plan.splits *
                                       (f.D + 2) * sizeof(float)
                                 : 0;
    } else {
        return f;
    }
    if (a->Hq <= 0 || a->Hq % f.Hkv != 0)
        return f;
    if (a->Hq / f.Hkv > 8) {
        f.st = KVC_ERR_UNSUPPORTED;
        return f;
    }
    f.st = KVC_OK;
    return f;
}

} // namespace
} // namespace kvc

using namespace kvc;

extern "C" {

size_t kvc_gear_side_bytes(int D)
{
    if (!head_dim_ok(D))
        return 0;
    const int ns = (2 * KIVI_G * D + 99) / 100;   // ceil(2% of the group's 32 x D entries)
    const int raw = 4 * ns + 4 * KIVI_G + 4 * D;   // indices, values, A [2][32], B [2][D]
    return (size_t)((raw + 15) / 16 * 16);
}

size_t kvc_kivi_block_bytes(int D, int bits)
{
    if (!head_dim_ok(D) || (bits != 2 && bits != 4))
        return 0;
    return (size_t)KIVI_G * D * bits / 8 + 4 * (size_t)D;
}

kvc_status kvc_append(const kvc_slot_cache *cache, const uint16_t *k_new, const uint16_t *v_new,
                      int n_new, cudaStream_t stream)
{
    kvc_status st = check_slot_cache(cache);
    if (st != KVC_OK)
        return st;
    if (n_new < 0 || (n_new > 0 && (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new))))
        return KVC_ERR_INVALID_ARG;
    if (n_new > cache->C)
        return KVC_ERR_CAPACITY;
    if (n_new == 0)
        return KVC_OK;
    return from_cuda(launch_append_slots(*cache, k_new, v_new, n_new, stream));
}

kvc_status kvc_append_quant(const kvc_quant_cache *cache, const uint16_t *k_new,
                            const uint16_t *v_new, int n_new, cudaStream_t stream)
{
    kvc_status st = check_quant_cache(cache);
    if (st != KVC_OK)
        return st;
    if (n_new < 0 || (n_new > 0 && (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new))))
        return KVC_ERR_INVALID_ARG;
    if (n_new == 0)
        return KVC_OK;
    if ((long long)n_new > (long long)cache->Cq + cache->R + KIVI_G)
        return KVC_ERR_CAPACITY;
    return from_cuda(launch_append_quant(*cache, k_new, v_new, n_new, stream));
}

size_t kvc_workspace_size(const kvc_attend_args *args)
{
    AttendPlanFull f = plan_full(args);
    return f.st == KVC_OK ? f.ws : 0;
}

kvc_status kvc_decode_attend(const kvc_attend_args *a, cudaStream_t stream)
{
    AttendPlanFull f = plan_full(a);
    if (f.st != KVC_OK)
        return f.st;
    if (!a->q || !a->o || !aligned16(a->q) || !aligned16(a->o))
        return KVC_ERR_INVALID_ARG;
    if (a->kind == KVC_KIND_KIVI && (a->logits || a->h2o_scores))
        return KVC_ERR_UNSUPPORTED;
    if (a->h2o_scores && !a->lse)
        return KVC_ERR_INVALID_ARG;
    float h2o_keep = 1.f, h2o_add = 1.f;
    if (!h2o_decay_weights(a->h2o_decay, &h2o_keep, &h2o_add))
        return KVC_ERR_INVALID_ARG;
    if (f.ws > 0 && (!a->workspace || a->workspace_bytes < f.ws || !aligned16(a->workspace)))
        return KVC_ERR_WORKSPACE;
    const float scale = a->softmax_scale > 0.f ? a->softmax_scale : 1.0f / sqrtf((float)f.D);
    float *part_o = static_cast<float *>(a->workspace);
    if (a->kind == KVC_KIND_SLOTS) {
        const kvc_slot_cache &c = *a->slots;
        float *part_ml = part_o ? part_o + (size_t)f.B * a->Hq * f.plan.splits * f.D : nullptr;
        AttendLaunch L{f.B, a->Hq, c.Hkv, c.D, c.C, a->q, a->o, c.K, c.V, c.n, a->logits, a->lse,
                       part_o, part_ml, f.plan.splits, f.plan.tiles_per_split, scale,
                       a->h2o_scores, h2o_keep, h2o_add, f.cluster, c.block_table, c.num_pages};
        cudaError_t e = launch_attend_slots(L, stream);
        if (e != cudaSuccess || !a->h2o_scores || f.plan.splits == 1 || f.cluster)
            return from_cuda(e);
        // several splits: the probabilities need the combined lse first
        kvc_h2o_args h{};
        h.mode = KVC_H2O_DECODE;
        h.B = f.B;
        h.Hq = a->Hq;
        h.Hkv = c.Hkv;
        h.D = c.D;
        h.C = c.C;
        h.scores = a->h2o_scores;
        h.logits = a->logits;
        h.lse = a->lse;
        h.n = c.n;
        h.decay = a->h2o_decay;
        return from_cuda(launch_h2o_decode_acc(h, stream));
    }
    const kvc_quant_cache &c = *a->quant;
    const size_t split_rows = (size_t)(f.B * f.Hkv - f.full_units) * (a->Hq / f.Hkv);
    float *part_ml = part_o ? part_o + split_rows * f.plan.splits * f.D : nullptr;
    KiviAttendLaunch L{f.B, a->Hq, c.Hkv, c.D, c.bits, c.R, c.Cq, a->q, a->o, c.k_blocks,
                       c.v_blocks, c.k_res, c.v_res, c.len, a->lse, part_o, part_ml,
                       f.plan.splits, f.plan.tiles_per_split, f.full_units, scale,
                       c.block_table, c.num_pages, c.k_gear, c.v_gear};
    return from_cuda(launch_attend_kivi(L, stream));
}

size_t kvc_h2o_workspace_size(const kvc_h2o_args *a)
{
    if (!a || a->mode != KVC_H2O_PREFILL || a->L <= 0 || a->B <= 0 || a->Hq <= 0)
        return 0;
    const size_t lpad = (size_t)((a->L + 127) / 128) * 128;   // whole 128-row query tiles
    // -lse of every prompt row, then the two passes' work counters (16 bytes)
    return (size_t)a->B * a->Hq * lpad * sizeof(float) + 16;
}

kvc_status kvc_h2o_accumulate(const kvc_h2o_args *a, cudaStream_t stream)
{
    if (!a || !a->scores || a->B <= 0 || a->Hkv <= 0 || a->Hq <= 0 || a->C <= 0)
        return KVC_ERR_INVALID_ARG;
    if (a->Hq % a->Hkv != 0)
        return KVC_ERR_INVALID_ARG;
    if (a->mode == KVC_H2O_DECODE) {
        float keep, add;
        if (!a->logits || !a->lse || !a->n || !h2o_decay_weights(a->decay, &keep, &add))
            return KVC_ERR_INVALID_ARG;
        return from_cuda(launch_h2o_decode_acc(*a, stream));
    }
    if (a->mode != KVC_H2O_PREFILL)
        return KVC_ERR_INVALID_ARG;
    if (!head_dim_ok(a->D))
        return KVC_ERR_UNSUPPORTED;
    if (!a->qp || !a->kp || a->L <= 0 || !aligned16(a->qp) || !aligned16(a->kp))
        return KVC_ERR_INVALID_ARG;
    if (a->L > a->kp_cap || a->L > a->C)
        return KVC_ERR_CAPACITY;
    if ((long long)a->B * a->Hq * a->L > (long long)INT_MAX ||
        (long long)a->B * a->Hkv * a->kp_cap > (long long)INT_MAX)
        return KVC_ERR_UNSUPPORTED;
    const size_t need = kvc_h2o_workspace_size(a);
    if (!a->workspace || a->workspace_bytes < need || !aligned16(a->workspace))
        return KVC_ERR_WORKSPACE;
    return from_cuda(launch_h2o_prefill(*a, static_cast<float *>(a->workspace), stream));
}

static kvc_status evict_common(const kvc_slot_cache *cache)
{
    kvc_status st = check_slot_cache(cache);
    if (st != KVC_OK)
        return st;
    if (cache->C > EVICT_MAX_SLOTS)
        return KVC_ERR_UNSUPPORTED;
    return KVC_OK;
}

kvc_status kvc_h2o_evict(const kvc_slot_cache *cache, float *scores, int n_heavy, int n_recent,
                         cudaStream_t stream)
{
    kvc_status st = evict_common(cache);
    if (st != KVC_OK)
        return st;
    if (!scores || n_heavy < 0 || n_recent < 0)
        return KVC_ERR_INVALID_ARG;
    EvictLaunch e{};
    e.kind = EVICT_H2O;
    e.c = *cache;
    e.scores = scores;
    e.n_heavy = n_heavy;
    e.n_recent = n_recent;
    return from_cuda(launch_evict(e, stream));
}

kvc_status kvc_h2o_evict_when(const kvc_slot_cache *cache, float *scores, int n_heavy,
                              int n_recent, int trigger, cudaStream_t stream)
{
    kvc_status st = evict_common(cache);
    if (st != KVC_OK)
        return st;
    if (!scores || n_heavy < 0 || n_recent < 0 || trigger <= 0)
        return KVC_ERR_INVALID_ARG;
    EvictLaunch e{};
    e.kind = EVICT_H2O;
    e.c = *cache;
    e.scores = scores;
    e.n_heavy = n_heavy;
    e.n_recent = n_recent;
    e.trigger = trigger;
    return from_cuda(launch_evict(e, stream));
}

kvc_status kvc_stream_evict(const kvc_slot_cache *cache, int n_sink, int n_recent,
                            cudaStream_t stream)
{
    kvc_status st = evict_common(cache);
    if (st != KVC_OK)
        return st;
    if (n_sink < 0 || n_recent < 0)
        return KVC_ERR_INVALID_ARG;
    EvictLaunch e{};
    e.kind = EVICT_STREAM;
    e.c = *cache;
    e.n_sink = n_sink;
    e.n_recent = n_recent;
    return from_cuda(launch_evict(e, stream));
}

static kvc_status decode_step_common(const kvc_slot_cache *cache, int Hq, const uint16_t *q,
                                     const uint16_t *k_new, const uint16_t *v_new, uint16_t *o,
                                     int n_recent, int n_other)
{
    kvc_status st = check_slot_cache(cache);
    if (st != KVC_OK)
        return st;
    if (!q || !o || !k_new || !v_new || !aligned16(q) || !aligned16(o) || !aligned16(k_new) ||
        !aligned16(v_new))
        return KVC_ERR_INVALID_ARG;
    if (Hq <= 0 || Hq % cache->Hkv != 0 || n_recent < 0 || n_other < 0)
        return KVC_ERR_INVALID_ARG;
    if (Hq / cache->Hkv > 8 || cache->Hkv > 127)
        return KVC_ERR_UNSUPPORTED;
    return KVC_OK;
}

kvc_status kvc_h2o_decode_step(const kvc_slot_cache *cache, float *scores, int Hq,
                               const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                               uint16_t *o, float *lse, int n_heavy, int n_recent, float decay,
                               cudaStream_t stream)
{
    kvc_status st = decode_step_common(cache, Hq, q, k_new, v_new, o, n_recent, n_heavy);
    if (st != KVC_OK)
        return st;
    if (!scores)
        return KVC_ERR_INVALID_ARG;
    if (cache->C > H2O_ONCHIP_MAX_SLOTS || cache->C % 4 != 0)
        return KVC_ERR_UNSUPPORTED;
    StepLaunch L{};
    L.c = *cache;
    L.Hq = Hq;
    L.q = q;
    L.o = o;
    L.lse = lse;
    L.k_new = k_new;
    L.v_new = v_new;
    L.scores = scores;
    if (!h2o_decay_weights(decay, &L.h2o_keep, &L.h2o_add))
        return KVC_ERR_INVALID_ARG;
    L.n_heavy = n_heavy;
    L.n_recent = n_recent;
    L.scale = 1.0f / sqrtf((float)cache->D);
    const int units = cache->B * cache->Hkv;
    if (units <= 4 * sm_count())
        return from_cuda(launch_decode_step(L, stream));
    // Many units (more than four per SM): the same step as three launches, append ->
    // attention with the fused score update (logits on chip, one split) -> eviction, which
    // measured faster there (the one-launch kernel's longer tail per CTA is not hidden over
    // many waves; at 4096 units 192 vs 201 us, at 256 units 25 vs 22 us in a CUDA graph)
    cudaError_t e = launch_append_slots(*cache, k_new, v_new, 1, stream);
    if (e == cudaSuccess) {
        AttendLaunch A{cache->B, Hq, cache->Hkv, cache->D, cache->C, q, o, cache->K, cache->V,
                       cache->n, nullptr, lse, nullptr, nullptr, 1, (cache->C + TILE - 1) / TILE,
                       L.scale, scores, L.h2o_keep, L.h2o_add, false, cache->block_table,
                       cache->num_pages};
        e = launch_attend_slots(A, stream);
    }
    if (e == cudaSuccess) {
        EvictLaunch ev{};
        ev.kind = EVICT_H2O;
        ev.c = *cache;
        ev.scores = scores;
        ev.n_heavy = n_heavy;
        ev.n_recent = n_recent;
        e = launch_evict(ev, stream);
    }
    return from_cuda(e);
}

kvc_status kvc_stream_decode_step(const kvc_slot_cache *cache, int Hq, const uint16_t *q,
                                  const uint16_t *k_new, const uint16_t *v_new, uint16_t *o,
                                  float *lse, int n_sink, int n_recent, cudaStream_t stream)
{
    kvc_status st = decode_step_common(cache, Hq, q, k_new, v_new, o, n_recent, n_sink);
    if (st != KVC_OK)
        return st;
    StepLaunch L{};
    L.c = *cache;
    L.Hq = Hq;
    L.q = q;
    L.o = o;
    L.lse = lse;
    L.k_new = k_new;
    L.v_new = v_new;
    L.n_sink = n_sink;
    L.n_recent = n_recent;
    L.scale = 1.0f / sqrtf((float)cache->D);
    return from_cuda(launch_decode_step(L, stream));
}

kvc_status kvc_stream_append(const kvc_slot_cache *cache, const uint16_t *k_new,
                             const uint16_t *v_new, int n_sink, int n_recent, cudaStream_t stream)
{
    kvc_status st = check_slot_cache(cache);
    if (st != KVC_OK)
        return st;
    if (n_sink < 0 || n_recent < 0 || !k_new || !v_new || !aligned16(k_new) || !aligned16(v_new))
        return KVC_ERR_INVALID_ARG;
    return from_cuda(launch_stream_append(*cache, k_new, v_new, n_sink, n_recent, stream));
}

kvc_status kvc_random_evict(const kvc_slot_cache *cache, int prompt_len, double keep_ratio,
                            uint64_t seed, uint32_t epoch, cudaStream_t stream)
{
    kvc_status st = evict_common(cache);
    if (st != KVC_OK)
        return st;
    if (prompt_len < 0 || !(keep_ratio >= 0.0 && keep_ratio <= 1.0))
        return KVC_ERR_INVALID_ARG;
    EvictLaunch e{};
    e.kind = EVICT_RANDOM;
    e.c = *cache;
    e.prompt_len = prompt_len;
    e.keep_ratio = keep_ratio;
    e.seed = seed;
    e.epoch = epoch;
    return from_cuda(launch_evict(e, stream));
}

const char *kvc_status_string(kvc_status s)
{
    switch (s) {
    case KVC_OK:
        return "KVC_OK";
    case KVC_ERR_INVALID_ARG:
        return "KVC_ERR_INVALID_ARG: null, misaligned or out-of-range argument";
    case KVC_ERR_UNSUPPORTED:
        return "KVC_ERR_UNSUPPORTED: shape or format outside what the kernels handle";
    case KVC_ERR_CAPACITY:
        return "KVC_ERR_CAPACITY: size exceeds a capacity";
    case KVC_ERR_WORKSPACE:
        return "KVC_ERR_WORKSPACE: workspace missing or too small";
    case KVC_ERR_CUDA:
        return "KVC_ERR_CUDA: a CUDA runtime call or launch failed";
    case KVC_ERR_DEVICE:
        return "KVC_ERR_DEVICE: a kernel flagged an inconsistent cache or an expired wait";
    }
    return "KVC_ERR_UNKNOWN";
}

kvc_status kvc_read_device_status(int *out, cudaStream_t stream)
{
    if (!out)
        return KVC_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(stream) != cudaSuccess)
        return KVC_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_status, sizeof(int)) != cudaSuccess)
        return KVC_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_status, &zero, sizeof(int)) != cudaSuccess)
        return KVC_ERR_CUDA;
    *out = v;
    return v ? KVC_ERR_DEVICE : KVC_OK;
}

} // extern "C"
