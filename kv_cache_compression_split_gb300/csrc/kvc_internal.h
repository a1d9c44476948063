// kvc_internal.h -- host-side glue shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/kvc.h"

namespace kvc {

constexpr int TILE = 64;           // tokens per pipeline stage of the decode kernels
constexpr int H2O_ONCHIP_MAX_SLOTS = KVC_H2O_ONCHIP_MAX_SLOTS;   // fused H2O, logits on chip
constexpr int KIVI_G = KVC_KIVI_GROUP;

// Device status word of the current device (set-up once per device).
int *dev_status_ptr();

// SM count of the current device.
int sm_count();

// Raise the dynamic shared-memory limit of kernel `func` to `bytes` on the current
// device, once per (kernel, device); thread safe.  Returns the attribute call's error.
cudaError_t set_smem_once(const void *func, int bytes);

// CTAs of `func` (threads per CTA, dynamic shared memory) resident on all SMs of the
// current device together (at least one per SM), cached per (kernel, device).
int resident_ctas(const void *func, int threads, int smem);

// cuTensorMapEncodeTiled through the runtime's driver entry point.
bool encode_tmap_2d_f16(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                        uint32_t box_inner, uint32_t box_rows);

struct SlotAttendPlan {
    int splits;
    int tiles_per_split;
};

// Split plan shared by kvc_workspace_size and kvc_decode_attend (at most
// max_splits splits when none are requested).
SlotAttendPlan plan_attend(int units, int tiles_per_unit, int requested_splits, int max_splits = 64);

// Splits of one unit that the slot attention merges inside a thread-block cluster.
constexpr int SLOT_CLUSTER_MAX = 8;

// ---- launchers (each returns a cudaError_t of the launch) ----

struct AttendLaunch {
    int B, Hq, Hkv, D, C;
    const uint16_t *q;
    uint16_t *o;
    const uint16_t *K, *V;
    const int32_t *n;
    float *logits, *lse;
    float *part_o, *part_ml;
    int splits, tiles_per_split;
    float scale;
    float *h2o_scores;
    float h2o_keep, h2o_add;   // scores = keep * scores + add * p
    bool cluster;              // 2..8 splits merged in a cluster (no workspace)
    const int32_t *block_table; // paged layout (nullptr: dense)
    int num_pages;
};
cudaError_t launch_attend_slots(const AttendLaunch &a, cudaStream_t s);

// One decode step of H2O (scores != nullptr) or StreamingLLM in one launch of the slot
// attention kernel (one split): the new token joins the attention and takes one slot.
struct StepLaunch {
    kvc_slot_cache c;
    int Hq;
    const uint16_t *q;
    uint16_t *o;
    float *lse;
    const uint16_t *k_new, *v_new;
    float *scores;
    float h2o_keep, h2o_add;
    int n_heavy, n_recent, n_sink;
    float scale;
};
cudaError_t launch_decode_step(const StepLaunch &a, cudaStream_t s);

struct KiviAttendLaunch {
    int B, Hq, Hkv, D, bits, R, Cq;
    const uint16_t *q;
    uint16_t *o;
    const uint8_t *kb, *vb;
    const uint16_t *k_res, *v_res;
    const int32_t *len;
    float *lse;
    float *part_o, *part_ml;
    int splits, tiles_per_split;
    int full_units;              // with splits > 1: units 0 .. full_units-1 run unsplit
    float scale;
    const int32_t *block_table;  // paged group blocks (nullptr: dense)
    int num_pages;
    const uint8_t *kg, *vg;      // GEAR side blocks (nullptr: KIVI)
};
cudaError_t launch_attend_kivi(const KiviAttendLaunch &a, cudaStream_t s);

// Merge the split partials of units unit0 .. unit0 + n_units - 1 (partial rows
// indexed from unit0) into o and lse.
cudaError_t launch_combine(int B, int Hq, int Hkv, int D, int splits, int unit0, int n_units,
                           const float *part_o, const float *part_ml, uint16_t *o, float *lse,
                           cudaStream_t s);

cudaError_t launch_append_slots(const kvc_slot_cache &c, const uint16_t *k_new,
                                const uint16_t *v_new, int n_new, cudaStream_t s);
cudaError_t launch_append_quant(const kvc_quant_cache &c, const uint16_t *k_new,
                                const uint16_t *v_new, int n_new, cudaStream_t s);
cudaError_t launch_stream_append(const kvc_slot_cache &c, const uint16_t *k_new,
                                 const uint16_t *v_new, int n_sink, int n_recent, cudaStream_t s);

// Weights of the decode score update scores = keep * scores + add * p for a
// decay of 0 (plain: 1, 1) or lambda in (0, 1) (lambda, 1 - lambda); false
// for any other decay.
bool h2o_decay_weights(float decay, float *keep, float *add);
cudaError_t launch_h2o_decode_acc(const kvc_h2o_args &a, cudaStream_t s);
// Two tcgen05 passes over the causal prompt; lse_ws holds B*Hq*ceil(L/128)*128 floats.
cudaError_t launch_h2o_prefill(const kvc_h2o_args &a, float *lse_ws, cudaStream_t s);

enum EvictKind { EVICT_H2O = 0, EVICT_STREAM = 1, EVICT_RANDOM = 2 };
struct EvictLaunch {
    EvictKind kind;
    kvc_slot_cache c;
    float *scores;
    int n_heavy, n_recent, n_sink, prompt_len;
    int trigger;   // H2O: only units with n >= trigger are evicted (0: all)
    double keep_ratio;
    uint64_t seed;
    uint32_t epoch;
};
cudaError_t launch_evict(const EvictLaunch &e, cudaStream_t s);

} // namespace kvc
