// h2o.cu -- H2O heavy-hitter score accumulation after a decode step
// ("Rethinking KV Cache Compression" guide, §2 and §16 "4 种方法逐步执行":
// H2O keeps the tokens with the largest accumulated attention).
//
// scores[b,hk,j] += sum_{h in group(hk)} exp(logit[b,h,j] - lse[b,h]) from the
// logits / lse that the decode attention wrote.  The prompt's scores come from
// the tensor-core prefill pass in h2o_prefill_tc.cu.
#include "kvc_device.cuh"
#include "kvc_internal.h"

#include <math.h>

namespace kvc {

namespace {

// ------------------------------------------------------------------ decode
// A thread per slot j of a unit.  The group's logits of slot j are loaded eight
// at a time before any is used, so each thread has its HBM reads in flight
// together (one read after another left the kernel at a third of the
// bandwidth); the sum runs over h = 0 .. g-1 in order.  Each probability is
// 2^(logit log2e - lse log2e), the form the attention's fused update uses.
constexpr int ACC_MAX_G = 8;
constexpr float LOG2E = 1.4426950408889634f;

__global__ void __launch_bounds__(256) k_h2o_decode_acc(int Hq, int Hkv, int C,
                                                        const float *__restrict__ logits,
                                                        const float *__restrict__ lse,
                                                        const int32_t *__restrict__ n,
                                                        float *__restrict__ scores, float keep,
                                                        float add, int *status)
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
    const size_t row0 = (size_t)b * Hq + (size_t)hk * g;
    float *sc = scores + (size_t)unit * C + j;
    const float old = *sc;
    float s = 0.f;
    for (int h0 = 0; h0 < g; h0 += ACC_MAX_G) {
        float x[ACC_MAX_G];
#pragma unroll
        for (int h = 0; h < ACC_MAX_G; ++h)
            x[h] = h0 + h < g ? logits[(row0 + h0 + h) * C + j] : 0.f;
#pragma unroll
        for (int h = 0; h < ACC_MAX_G; ++h)
            if (h0 + h < g)
                s += ex2(fmaf(x[h], LOG2E, -lse[row0 + h0 + h] * LOG2E));
    }
    *sc = fmaf(old, keep, s * add);
}

// The same update, four consecutive slots per thread with 16-byte loads and
// stores (rows of C floats with C a multiple of 4, 16-byte aligned arrays):
// a quarter of the threads and load instructions, each slot's sum unchanged.
__global__ void __launch_bounds__(128) k_h2o_decode_acc4(int Hq, int Hkv, int C,
                                                         const float *__restrict__ logits,
                                                         const float *__restrict__ lse,
                                                         const int32_t *__restrict__ n,
                                                         float *__restrict__ scores, float keep,
                                                         float add, int *status)
{
    const int unit = blockIdx.x;
    const int b = unit / Hkv, hk = unit % Hkv, g = Hq / Hkv;
    int nn = n[unit];
    if (nn > C) {
        if (blockIdx.y == 0 && threadIdx.x == 0)
            flag_error(status, DEV_CAPACITY);
        nn = C;
    }
    const int j = 4 * (blockIdx.y * blockDim.x + threadIdx.x);
    if (j >= nn)
        return;
    // j + 3 < C: the slots past nn in this quad are read, not written
    const size_t row0 = (size_t)b * Hq + (size_t)hk * g;
    float *sc = scores + (size_t)unit * C + j;
    const float4 old = *reinterpret_cast<const float4 *>(sc);
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
    for (int h0 = 0; h0 < g; h0 += ACC_MAX_G) {
        float4 x[ACC_MAX_G];
        float l[ACC_MAX_G];
#pragma unroll
        for (int h = 0; h < ACC_MAX_G; ++h) {
            if (h0 + h < g) {
                x[h] = *reinterpret_cast<const float4 *>(logits + (row0 + h0 + h) * C + j);
                l[h] = lse[row0 + h0 + h] * LOG2E;
            }
        }
#pragma unroll
        for (int h = 0; h < ACC_MAX_G; ++h) {
            if (h0 + h < g) {
                s0 += ex2(fmaf(x[h].x, LOG2E, -l[h]));
                s1 += ex2(fmaf(x[h].y, LOG2E, -l[h]));
                s2 += ex2(fmaf(x[h].z, LOG2E, -l[h]));
                s3 += ex2(fmaf(x[h].w, LOG2E, -l[h]));
            }
        }
    }
    const float4 r = make_float4(fmaf(old.x, keep, s0 * add), fmaf(old.y, keep, s1 * add),
                                 fmaf(old.z, keep, s2 * add), fmaf(old.w, keep, s3 * add));
    if (j + 3 < nn) {
        *reinterpret_cast<float4 *>(sc) = r;
    } else {
        sc[0] = r.x;
        if (j + 1 < nn)
            sc[1] = r.y;
        if (j + 2 < nn)
            sc[2] = r.z;
    }
}

} // namespace

bool h2o_decay_weights(float decay, float *keep, float *add)
{
    if (decay == 0.f) {
        *keep = 1.f;
        *add = 1.f;
        return true;
    }
    if (decay > 0.f && decay < 1.f) {
        *keep = decay;
        *add = 1.f - decay;   // exact for decay in [0.5, 1)
        return true;
    }
    return false;
}

cudaError_t launch_h2o_decode_acc(const kvc_h2o_args &a, cudaStream_t s)
{
    float keep = 1.f, add = 1.f;
    if (!h2o_decay_weights(a.decay, &keep, &add))
        return cudaErrorInvalidValue;
    const bool vec = a.C % 4 == 0 && ((reinterpret_cast<uintptr_t>(a.logits) |
                                       reinterpret_cast<uintptr_t>(a.scores)) & 15u) == 0;
    if (vec) {
        dim3 grid(a.B * a.Hkv, (a.C / 4 + 127) / 128);
        k_h2o_decode_acc4<<<grid, 128, 0, s>>>(a.Hq, a.Hkv, a.C, a.logits, a.lse, a.n, a.scores,
                                               keep, add, dev_status_ptr());
    } else {
        dim3 grid(a.B * a.Hkv, (a.C + 255) / 256);
        k_h2o_decode_acc<<<grid, 256, 0, s>>>(a.Hq, a.Hkv, a.C, a.logits, a.lse, a.n, a.scores,
                                              keep, add, dev_status_ptr());
    }
    return cudaGetLastError();
}

} // namespace kvc
