/*
 * kvc.h -- C ABI of the GB300 compressed-KV decode library (libkvc.so).
 *
 * One decode-attention step over a compressed KV cache, plus the cache
 * compression operators that keep the cache within budget:
 *   - KIVI asymmetric group quantisation (K per channel, V per token, groups of
 *     32, newest R tokens kept in fp16)       -- kvc_append_quant
 *   - split-KV decode attention over an fp16 slot cache or a KIVI cache, with
 *     GQA head mapping                        -- kvc_decode_attend
 *   - H2O heavy-hitter scores and eviction    -- kvc_h2o_accumulate, kvc_h2o_evict
 *   - whole decode steps in one launch        -- kvc_h2o_decode_step,
 *                                                kvc_stream_decode_step
 *   - StreamingLLM sink + recent window       -- kvc_stream_evict, kvc_stream_append
 *   - per-head uniform random eviction with the prompt locked
 *                                             -- kvc_random_evict
 *
 * Method sources (web pages, cited by title and section):
 *   "Rethinking KV Cache Compression: 从显存节省回到真实 serving 端到端收益"
 *     (guide), §2 "4 种 baseline 的成本结构" (KIVI G=32, R=128; StreamingLLM and
 *     H2O keep 64 initial / heavy + 448 recent = 512), §16 "4 种方法逐步执行"
 *     (KIVI per-channel K and per-token V with a full-precision residual,
 *     dequantised on the decode read; StreamingLLM keeps sinks and the recent
 *     window; H2O accumulates attention and updates its keep set) and §16
 *     "局限与最终结论" (old tokens are converted when the residual fills; the
 *     H2O score needs attention probabilities that flash attention does not
 *     materialise, hence the extra prefill pass).
 *   "KV Cache 驱逐实战：什么时候该放弃打分器，直接随机扔", section "参考实现"
 *     (per-head uniform random eviction with the prompt locked; every head
 *     keeps the same count, prompt_len + n_keep, never a union over heads).
 *   "Practical Online KV Cache Compaction for LLM Agents" (demingchina.com),
 *     §4.2 (mark the dropped entries, compact the kept ones, keep a
 *     logical -> physical position map): the slot caches below are compacted
 *     in place and carry each slot's absolute position.
 *
 * Conventions for every call
 *   - All pointers inside the descriptors are DEVICE pointers owned by the
 *     caller; the library allocates nothing and keeps no state other than one
 *     device status word per GPU.  Every call is asynchronous on `stream` and
 *     returns after enqueueing its kernels.
 *   - fp16 means IEEE binary16, passed as uint16_t bit patterns.  All data
 *     must be finite.  Pointers must be 16-byte aligned.
 *   - Head dim D is 64 or 128; Hq is a multiple of Hkv with 1 <= Hq/Hkv <= 8;
 *     query head h reads KV head h / (Hq/Hkv).  Softmax scale defaults to
 *     1/sqrt(D).
 *   - Argument errors are reported synchronously and enqueue nothing.  Errors
 *     that depend on device-resident counts (a count above capacity, a wait
 *     that ran out) set the device status word; the kernel then skips the
 *     offending unit and the cache contents of that unit are unspecified.
 *     Read (and clear) it with kvc_read_device_status.  No kernel traps.
 */
#ifndef KVC_H
#define KVC_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define KVC_API __attribute__((visibility("default")))
#else
#define KVC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvc_status {
    KVC_OK = 0,
    KVC_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned pointer */
    KVC_ERR_UNSUPPORTED = 2, /* D, bits, group ratio outside what the kernels handle */
    KVC_ERR_CAPACITY = 3,    /* a size the host can check exceeds a capacity */
    KVC_ERR_WORKSPACE = 4,   /* workspace missing or smaller than kvc_workspace_size */
    KVC_ERR_CUDA = 5,        /* a CUDA runtime call or kernel launch failed */
    KVC_ERR_DEVICE = 6       /* returned by kvc_read_device_status when a kernel flagged an error */
} kvc_status;

/* Device status word bits (kvc_read_device_status). */
#define KVC_DEV_CAPACITY 0x1 /* a device-resident count exceeded its capacity */
#define KVC_DEV_TIMEOUT 0x2  /* a bounded wait on a shared-memory barrier ran out */

/* KIVI group size (tokens per K group, channels per V group). */
#define KVC_KIVI_GROUP 32

/*
 * Slot cache: the fp16 cache used by full attention, H2O, StreamingLLM and
 * random eviction.  Each (b, kv_head) unit owns C slots; slots [0, n[b,h])
 * are valid and hold the tokens whose absolute positions are in pos[].
 * Slot order is free (attention does not depend on it); evictions compact the
 * kept slots into [0, n') by moving kept slots from the tail into the holes.
 *   K, V   [B, Hkv, C, D] fp16 (dense layout), or page pools (paged layout)
 *   pos    [B, Hkv, C]    int32, absolute token position of each slot
 *   n      [B, Hkv]       int32, valid slots of each unit
 *   seqlen [B]            int32, tokens generated so far by sequence b (the
 *                         absolute position the next appended token gets)
 *   block_table  NULL for the dense layout.  Paged layout: [B, Hkv, C / 64]
 *                int32; slot j of unit (b, h) is row j % 64 of page
 *                block_table[b][h][j / 64], and K, V are pools of
 *                [num_pages, 64, D] fp16 shared by all units.  C must be a
 *                multiple of KVC_PAGE_SLOTS.  The caller owns the pool and the
 *                table: every slot a call writes must map to a page in
 *                [0, num_pages) that no other unit uses (entries of slots
 *                beyond a unit's pages may be -1, so units of a ragged batch
 *                hold only the pages they need).  A write through an entry
 *                outside [0, num_pages) is skipped and sets KVC_DEV_CAPACITY.
 *   num_pages    pages in each pool (paged layout only)
 * The paged layout is the block layout of paged attention, which splits the
 * cache into blocks so that it can be allocated non-contiguously and batched
 * continuously ("Rethinking KV Cache Compression" guide, §16 "前置背景、复现方法
 * 与结论边界"); here every (sequence, KV head) unit has its own page list because
 * the eviction methods compact each head on its own.
 */
#define KVC_PAGE_SLOTS 64
typedef struct kvc_slot_cache {
    int B, Hkv, D, C;
    uint16_t *K;
    uint16_t *V;
    int32_t *pos;
    int32_t *n;
    int32_t *seqlen;
    const int32_t *block_table;
    int num_pages;
} kvc_slot_cache;

/*
 * KIVI cache.  For a sequence of T = len[b] tokens the first
 *   n_q = 32 * floor(max(0, T - R) / 32)
 * tokens are held quantised and tokens [n_q, T) are held in fp16 in a ring of
 * R + 32 slots (token p in slot p mod (R + 32)).  Group g covers tokens
 * [32 g, 32 g + 32).  Quantisation of a group of values x (asymmetric):
 *   zero  = min(x) (binary16; a zero minimum is stored as +0)
 *   scale = binary16 round-to-nearest-even of (max(x) - min(x)) / (2^bits - 1)
 *   code  = clamp(round-half-even((x - zero) / scale), 0, 2^bits - 1), computed
 *           exactly; a group with scale 0 gets codes 0
 *   value = zero + code * scale
 * K is grouped per channel over the 32 tokens of a group; V is grouped per
 * token over 32 consecutive channels.
 *
 * Block layout (k_blocks and v_blocks are [B, Hkv, Cq/32, block_bytes] bytes,
 * block_bytes = 32*D*bits/8 + 4*D, see kvc_kivi_block_bytes):
 *   K block: 32 token rows of WK = D*bits/32 little-endian u32 words; in token
 *     t's word w, field i (bits [bits*i, bits*(i+1))) holds channel
 *     d = (32/bits)*w + i.  Then D fp16 scales (per channel), then D fp16 zeros.
 *   V block: 16 token pairs of 2*WK words.  Pair i holds tokens 2i (low 16 bits
 *     of every word) and 2i+1 (high 16 bits).  Its word ((r + 2i) mod 8)*W + k
 *     (r in [0,8), k in [0,W), W = D*bits/128) holds in field j (bits
 *     [bits*j, bits*(j+1)) of each 16-bit half) channel
 *     d = 16*(k*(8/bits) + j/2) + 8*(j%2) + r.
 *     Then the V scales as D/32 rows of 32 fp16 values (row j holds channel
 *     group j of tokens 0..31), then the V zeros in the same [D/32][32] order.
 *   k_res, v_res [B, Hkv, R + 32, D] fp16 residual rings;  len [B] int32.
 *   block_table  NULL for the dense layout above.  Paged layout: pages of
 *                KVC_KIVI_PAGE_GROUPS = 4 consecutive groups (128 tokens);
 *                group g of unit (b, h) is block g % 4 of page
 *                block_table[b][h][g / 4] ([B, Hkv, Cq / 128] int32) in
 *                k_blocks / v_blocks pools of [num_pages, 4, block_bytes].
 *                Cq must be a multiple of 128; the ownership and error rules
 *                are those of the paged slot cache (entries of pages a unit
 *                does not use may be -1; a write through an entry outside
 *                [0, num_pages) is skipped and sets KVC_DEV_CAPACITY, and a
 *                read through one yields no data for that tile).
 *   num_pages    pages in each pool (paged layout only)
 *   k_gear, v_gear  NULL for KIVI.  GEAR: per group one side block of
 *                kvc_gear_side_bytes(D) bytes, [B, Hkv, Cq/32, side_bytes] (paged
 *                layout: pools [num_pages, 4, side_bytes], group g of a unit at
 *                the same page and slot as its K / V block), holding a 2% sparse
 *                and a rank-2 correction of the
 *                group's quantisation residual ("Rethinking KV Cache Compression"
 *                guide, §2: GEAR sparsity 2%, rank 2; §16: the corrections act on
 *                KIVI's quantisation residual).  With x_q = fl32(zero + code *
 *                scale) and the fp32 residual e = fl32(x - x_q) of every element:
 *                  n_s = ceil(2% * 32 * D) u16 flat indices t*D + d (ascending) of
 *                    the entries with the largest |e| (ties: lower index), then
 *                    their binary16 values RN16(e);
 *                  A [2][32] binary16: orthonormal rows spanning the dominant
 *                    2-dimensional left singular subspace of R = E with the
 *                    sparse entries zeroed; B [2][D] binary16 = A R;
 *                  zero padding to a multiple of 16 bytes.
 *                Decode attention then uses x_hat = x_q + S + A^T B for the
 *                quantised tokens.
 */
#define KVC_KIVI_PAGE_GROUPS 4
typedef struct kvc_quant_cache {
    int B, Hkv, D, bits, R, Cq; /* Cq: quantised-token capacity, a multiple of 32 */
    uint8_t *k_blocks;
    uint8_t *v_blocks;
    uint16_t *k_res;
    uint16_t *v_res;
    int32_t *len;
    const int32_t *block_table;
    int num_pages;
    uint8_t *k_gear;
    uint8_t *v_gear;
} kvc_quant_cache;

/* Bytes of one K (or V) block: 32*D*bits/8 + 4*D. */
KVC_API size_t kvc_kivi_block_bytes(int D, int bits);

/* Bytes of one GEAR side block (see kvc_quant_cache): 976 for D = 128, 560 for
 * D = 64, 0 for an unsupported D. */
KVC_API size_t kvc_gear_side_bytes(int D);

/*
 * kvc_append -- write n_new tokens per sequence into a slot cache.
 * Rows [B, Hkv, n_new, D] of k_new / v_new (fp16, device) go to slots
 * n[b,h] .. n[b,h]+n_new-1 with positions seqlen[b] .. seqlen[b]+n_new-1;
 * then n += n_new and seqlen += n_new.  A unit that would exceed C sets
 * KVC_DEV_CAPACITY and is left unchanged.
 * Source: the KV cache keeps every generated token's K/V per layer
 * ("Rethinking KV Cache Compression" guide, §16 "KV cache 的容量公式").
 */
KVC_API kvc_status kvc_append(const kvc_slot_cache *cache, const uint16_t *k_new, const uint16_t *v_new,
                      int n_new, cudaStream_t stream);

/*
 * kvc_append_quant -- append n_new tokens per sequence to a KIVI cache.
 * New tokens enter the fp16 residual; every group of 32 that leaves the
 * residual window (see n_q above) is quantised and packed.  k_new / v_new are
 * [B, Hkv, n_new, D] fp16.  Then len += n_new.  n_q above Cq sets
 * KVC_DEV_CAPACITY for that unit.
 * Source: "Rethinking KV Cache Compression" guide, §2 (G=32, R=128), §16 "4 种
 * 方法逐步执行" and "局限与最终结论" (the residual converts when full).
 */
KVC_API kvc_status kvc_append_quant(const kvc_quant_cache *cache, const uint16_t *k_new,
                            const uint16_t *v_new, int n_new, cudaStream_t stream);

enum { KVC_KIND_SLOTS = 0, KVC_KIND_KIVI = 1 };

/*
 * Decode attention arguments.
 *   kind        KVC_KIND_SLOTS (fp16 slot cache) or KVC_KIND_KIVI
 *   Hq          query heads (a multiple of the cache's Hkv, at most 8 per KV head)
 *   q           [B, Hq, D] fp16, one query per sequence
 *   o           [B, Hq, D] fp16 output, o = sum_j softmax_j(scale q.k_j) v_j
 *   slots/quant the cache (the other pointer may be NULL)
 *   logits      optional [B, Hq, C] fp32 (slot caches only): scale * q.k_j of
 *               every valid slot j, in slot order (H2O decode scores)
 *   lse         optional [B, Hq] fp32: log sum_j exp(scale q.k_j); -inf for an
 *               empty unit (whose output is 0)
 *   workspace   device scratch of at least kvc_workspace_size(args) bytes
 *               (may be NULL when that size is 0)
 *   num_splits  KV splits per unit (0 = chosen from the SM count)
 *   softmax_scale 0 for 1/sqrt(D)
 *   h2o_scores  optional [B, Hkv, C] fp32 (slot caches only; needs lse): the
 *               step's attention probabilities are folded into the heavy-hitter
 *               scores in the same launch, exactly as
 *               kvc_h2o_accumulate(KVC_H2O_DECODE) with decay h2o_decay would.
 *               With logits NULL the launch keeps the logits on chip, each
 *               split its own: it then runs in at most 8 splits (a larger
 *               num_splits is KVC_ERR_INVALID_ARG) of at most
 *               KVC_H2O_ONCHIP_MAX_SLOTS slots each (else KVC_ERR_UNSUPPORTED);
 *               up to 576 slots per split the logits stay in registers, beyond
 *               that in shared memory (fewer pipeline stages).  With 2 to 8
 *               splits (logits on chip or not) the splits of a unit run as one
 *               thread-block cluster that merges them on chip and updates the
 *               scores in the same launch; with more splits (a logits array is
 *               then needed) the scores are updated by one kvc_h2o_accumulate
 *               launch after the combine.  For the same split count all
 *               storage modes give bit-identical o, lse and scores.
 *   h2o_decay   0 (plain H2O, scores += p) or lambda in (0, 1) (decayed
 *               scores = lambda * scores + (1 - lambda) * p); see kvc_h2o_args
 */
#define KVC_H2O_ONCHIP_MAX_SLOTS 1024
typedef struct kvc_attend_args {
    int kind;
    int Hq;
    const uint16_t *q;
    uint16_t *o;
    const kvc_slot_cache *slots;
    const kvc_quant_cache *quant;
    float *logits;
    float *lse;
    void *workspace;
    size_t workspace_bytes;
    int num_splits;
    float softmax_scale;
    float *h2o_scores;
    float h2o_decay;
} kvc_attend_args;

/* Workspace bytes kvc_decode_attend needs for these arguments (0 if none). */
KVC_API size_t kvc_workspace_size(const kvc_attend_args *args);

/*
 * kvc_decode_attend -- one decode step of attention over the compressed cache.
 * Every (sequence, KV head) unit is split along the cache into num_splits
 * ranges; each range keeps a running max / sum / weighted value sum (flash
 * decoding), and a combine step merges the ranges.  KIVI caches are
 * dequantised in registers: the per-channel K scale is folded into the query
 * per group and the per-token V scale into the probabilities; the fp16
 * residual tail is attended in the same pass.  A KIVI cache with GEAR side
 * blocks (k_gear, v_gear) is attended over x_q + S + A^T B: the sparse and
 * rank-2 corrections are applied in the same kernel (GEAR: "Rethinking KV
 * Cache Compression" guide, §2, sparsity 2%, rank 2).
 * Source: "Rethinking KV Cache Compression" guide, §16 "Prefill、decode、TP 的
 * 性能账" (decode reads all history and is bandwidth bound) and "4 种方法逐步
 * 执行" (KIVI dequantises on the decode read).
 */
KVC_API kvc_status kvc_decode_attend(const kvc_attend_args *args, cudaStream_t stream);

/* Size of the library-owned scratch array used by kvc_decode_attend_noalloc. */
#define KVC_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * kvc_decode_attend_noalloc -- kvc_decode_attend for callers that cannot
 * allocate device memory on their decode path (for example a serving engine
 * that gives all free device memory to its KV-cache pool at start-up, or a
 * plugin host that forbids cudaMalloc / cudaFree in its enqueue callback
 * because they synchronise the device).  The pages describe no such variant;
 * it is an interface convenience of this library.
 *
 * Same arguments and results as kvc_decode_attend, except that args->workspace
 * and args->workspace_bytes are ignored: the split scratch comes from one
 * fixed device array of KVC_NOALLOC_SCRATCH_BYTES that the library owns (held
 * by every GPU that loads the library until the process exits).  The call
 * allocates nothing.  Arguments whose kvc_workspace_size exceeds
 * KVC_NOALLOC_SCRATCH_BYTES are rejected with KVC_ERR_WORKSPACE.
 * The first call on a device that needs scratch looks up that array's device
 * address (cudaGetSymbolAddress) with the device current and keeps it; make
 * that first call before any stream capture.  The kept address belongs to the
 * device code loaded at that time: do not call this entry point after a
 * cudaDeviceReset.  All calls on a device share the array, so calls whose
 * kernels may overlap on the GPU (unordered streams) race; order them.
 */
KVC_API kvc_status kvc_decode_attend_noalloc(const kvc_attend_args *args, cudaStream_t stream);

enum { KVC_H2O_DECODE = 0, KVC_H2O_PREFILL = 1 };

/*
 * H2O score arguments.
 *   scores   [B, Hkv, C] fp32, one accumulated score per slot
 * DECODE:  p[b,hk,j] = sum over the query heads h of KV head hk of
 *          exp(logits[b,h,j] - lse[b,h]) for j < n[b,hk]  (logits, lse from
 *          kvc_decode_attend; n [B, Hkv]), then
 *            decay == 0:          scores[b,hk,j] += p[b,hk,j]
 *            0 < decay < 1:       scores[b,hk,j] = decay * scores[b,hk,j]
 *                                                  + (1 - decay) * p[b,hk,j]
 *          The decayed form is the incremental activity score
 *          A_i <- lambda A_i + (1 - lambda) attn_i (lambda = 0.99 on the page) of
 *          "Practical Online KV Cache Compaction for LLM Agents", §4.1; PREFILL
 *          ignores decay.
 * PREFILL: scores[b,hk,j] = sum over the query heads h of hk, and over prompt
 *          rows i >= j, of softmax_i(scale * qp[b,h,i] . kp[b,hk,.])_j for
 *          j < L (causal prompt of L tokens); qp [B, Hq, L, D] fp16, kp the
 *          prompt keys [B, Hkv, kp_cap, D] fp16 with prompt token j in row j.
 *          Needs kvc_h2o_workspace_size bytes of workspace (16-byte aligned):
 *          -lse of every prompt row ([B * Hq, L rounded up to 128] fp32), then
 *          16 bytes of work counters that the call zeroes on its stream.
 *          lse (optional): [B, Hq, L] fp32, each prompt row's natural-log
 *          normaliser log sum_{j <= i} exp(scale * qp[b,h,i] . kp[b,hk,j]), as a
 *          causal flash-attention forward over the same prompt returns it.
 *          When given, the pass that computes these is skipped and only the
 *          column-sum pass runs (the one extra pass over the prompt); when NULL
 *          the call computes them itself.  The values are read as given.
 */
typedef struct kvc_h2o_args {
    int mode;
    int B, Hq, Hkv, D, C;
    float *scores;
    const float *logits;
    const float *lse;
    const int32_t *n;
    int L;
    const uint16_t *qp;
    const uint16_t *kp;
    int kp_cap;
    void *workspace;
    size_t workspace_bytes;
    float softmax_scale;
    float decay;
} kvc_h2o_args;

KVC_API size_t kvc_h2o_workspace_size(const kvc_h2o_args *args);

/*
 * kvc_h2o_accumulate -- add attention probabilities into the heavy-hitter
 * scores (DECODE) or compute the prompt's scores in a second pass over the
 * causal prompt (PREFILL: one pass for the row log-sum-exp, unless the caller
 * supplies it, and one that recomputes the probabilities and sums them per
 * key).
 * Source: "Rethinking KV Cache Compression" guide, §16 "4 种方法逐步执行" (H2O
 * accumulates attention scores) and "局限与最终结论" (the extra pass).
 */
KVC_API kvc_status kvc_h2o_accumulate(const kvc_h2o_args *args, cudaStream_t stream);

/*
 * kvc_h2o_evict -- per unit keep the recent window (positions >= seqlen[b] -
 * n_recent) and the n_heavy other slots with the largest scores (ties: lower
 * position first); compact K, V, pos and scores [B, Hkv, C] and set n.  The
 * scores of the freed slots [n', n) are set to 0, so a token appended there
 * later starts from a zero score (new slots beyond the old n must be 0 too:
 * zero the whole scores array when the cache is created).
 * A unit with at most n_heavy + n_recent slots is unchanged.
 * Source: "Rethinking KV Cache Compression" guide, §2 (64 heavy + 448 recent)
 * and §16 "4 种方法逐步执行".
 */
KVC_API kvc_status kvc_h2o_evict(const kvc_slot_cache *cache, float *scores, int n_heavy, int n_recent,
                         cudaStream_t stream);

/*
 * kvc_h2o_evict_when -- batched H2O eviction: exactly kvc_h2o_evict for the
 * units with n[b,hk] >= trigger; every other unit is left unchanged.  With
 * trigger = 1.1 x (n_heavy + n_recent) a unit is compacted once every ~10% of
 * the budget in new tokens instead of at every step ("Practical Online KV
 * Cache Compaction for LLM Agents", §5.2: compact when the cache passes 110% of
 * its target, or every K = 50 tokens).  The check runs on the device, so the
 * call never reads n back and can sit in a captured graph.  trigger must be
 * > 0; a trigger at or below n_heavy + n_recent is kvc_h2o_evict.
 */
KVC_API kvc_status kvc_h2o_evict_when(const kvc_slot_cache *cache, float *scores, int n_heavy,
                              int n_recent, int trigger, cudaStream_t stream);

/*
 * kvc_stream_evict -- StreamingLLM: keep positions < n_sink and positions
 * >= seqlen[b] - n_recent; compact and set n.
 * Source: "Rethinking KV Cache Compression" guide, §2 (64 sinks + 448 recent)
 * and §16 "4 种方法逐步执行".
 */
KVC_API kvc_status kvc_stream_evict(const kvc_slot_cache *cache, int n_sink, int n_recent,
                            cudaStream_t stream);

/*
 * kvc_stream_append -- StreamingLLM decode step without an eviction launch.
 * Appends one token per sequence (k_new / v_new [B, Hkv, 1, D] fp16, device) at
 * position P = seqlen[b], then seqlen += 1.  In each unit, the token that leaves
 * the window with this step -- position P - n_recent - 1, when that is >= n_sink --
 * gives up its slot: the new token overwrites that slot's K, V and position and n
 * is unchanged.  When no valid slot holds that position the token goes to slot n
 * and n += 1 (a unit at capacity sets KVC_DEV_CAPACITY and is left unchanged).
 * So a unit that holds the window of the previous step ([0, n_sink) and
 * [P - 1 - n_recent, P - 1]), or the keep set of kvc_stream_evict after the
 * prompt, holds after the call exactly this step's attention window
 *   positions < n_sink  and  P - n_recent <= position <= P
 * (n_sink + n_recent + 1 tokens in steady state).  The step's decode attention
 * then reads that window, and the token that left it is dropped by the next
 * call's overwrite, with no scan-and-move launch: the eviction is metadata only.
 * The attention sets are those of append -> attend -> kvc_stream_evict.
 * Source: "Rethinking KV Cache Compression" guide, §2 (64 sinks + 448 recent)
 * and §16 "4 种方法逐步执行" (sinks plus the recent window, no scores).
 */
KVC_API kvc_status kvc_stream_append(const kvc_slot_cache *cache, const uint16_t *k_new,
                             const uint16_t *v_new, int n_sink, int n_recent,
                             cudaStream_t stream);

/*
 * kvc_h2o_decode_step -- one H2O decode step in one launch: append, attention with
 * the heavy-hitter score update, and the eviction back to n_heavy + n_recent.
 * The same results as kvc_append (k_new / v_new [B, Hkv, 1, D] fp16, position
 * P = seqlen[b]) -> kvc_decode_attend (o [B, Hq, D], lse [B, Hq] optional, with
 * h2o_scores = scores and h2o_decay = decay) -> kvc_h2o_evict(n_heavy, n_recent),
 * for caches whose units hold at most n_heavy + n_recent slots before the step (the
 * decode steady state: at most one slot leaves per step).  The new token attends
 * from k_new / v_new; afterwards at most one K/V row is written: into the slot
 * that leaves (the worst non-recent slot by score descending, position
 * ascending), with its score set to the new token's, or into slot n while the
 * unit is below budget (n += 1); with n_recent = 0 the new token itself may be
 * the one that leaves, and then nothing is written.  seqlen += 1.  One split per
 * unit; C at most KVC_H2O_ONCHIP_MAX_SLOTS and a multiple of 4 (else
 * KVC_ERR_UNSUPPORTED); Hkv at most 127; positions below 2^24 - 1.  For batches
 * of more than four units per SM the call issues the three launches instead
 * (append, attention with the fused update, eviction; the results are the same),
 * which measured faster there.  A unit above budget is outside the contract: the
 * one-launch form sets KVC_DEV_CAPACITY and
 * keeps its slots (its o, lse and scores are still written).  While the kernel
 * runs, seqlen[b] carries an arrival count in its top 8 bits: nothing else may
 * read it concurrently.
 * Source: "Rethinking KV Cache Compression" guide, §2 (64 heavy + 448 recent) and
 * §16 "4 种方法逐步执行" (accumulate attention, update the keep set).
 */
KVC_API kvc_status kvc_h2o_decode_step(const kvc_slot_cache *cache, float *scores, int Hq,
                               const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                               uint16_t *o, float *lse, int n_heavy, int n_recent, float decay,
                               cudaStream_t stream);

/*
 * kvc_stream_decode_step -- one StreamingLLM decode step in one launch: the same
 * results as kvc_stream_append -> kvc_decode_attend (o, lse optional).  The token
 * that left the window with the previous step (position P - n_recent - 1, when
 * >= n_sink) is not attended and its slot takes the new token after the attention;
 * otherwise the token goes to slot n (n += 1).  seqlen += 1.  One split per unit;
 * Hkv at most 127; positions below 2^24 - 1; the seqlen arrival count of
 * kvc_h2o_decode_step applies.
 * Source: "Rethinking KV Cache Compression" guide, §2 (64 sinks + 448 recent) and
 * §16 "4 种方法逐步执行".
 */
KVC_API kvc_status kvc_stream_decode_step(const kvc_slot_cache *cache, int Hq, const uint16_t *q,
                                  const uint16_t *k_new, const uint16_t *v_new, uint16_t *o,
                                  float *lse, int n_sink, int n_recent, cudaStream_t stream);

/*
 * kvc_random_evict -- per-head uniform random eviction with the prompt locked.
 * Per unit (b, h): slots with pos < prompt_len stay; of the n_cand others keep
 * n_keep = max(1, (int)(n_cand * keep_ratio)), the n_keep with the smallest
 * 64-bit keys key = (w0 << 32) | w1 of Philox4x32-10 (Salmon et al., SC'11)
 * with key words (seed & 0xffffffff, seed >> 32) and counter
 * (pos, h, b, epoch) (ties: lower position).  Each head draws its own set and
 * every head keeps the same count; nothing is ever united across heads.
 * n_cand == 0 is a no-op.  keep_ratio must be in [0, 1].
 * Source: "KV Cache 驱逐实战" (tuntang.top), section "参考实现".
 */
KVC_API kvc_status kvc_random_evict(const kvc_slot_cache *cache, int prompt_len, double keep_ratio,
                            uint64_t seed, uint32_t epoch, cudaStream_t stream);

/* Human-readable name of a status code (static storage). */
KVC_API const char *kvc_status_string(kvc_status status);

/*
 * kvc_read_device_status -- synchronise `stream`, copy the current device's
 * status word into *out (KVC_DEV_* bits, 0 if clean) and clear it.  Returns
 * KVC_ERR_DEVICE if any bit was set, KVC_OK otherwise.
 */
KVC_API kvc_status kvc_read_device_status(int *out, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H */
