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
__global__ void k_h2o_decode_acc(int Hq, int Hkv, int C, const float *__restrict__ logits,
                                 const float *__restrict__ lse, const int32_t *__restrict__ n,
                                 float *__restrict__ scores, float keep, float add, int *status)
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
    float s = 0.f;
    for (int h = 0; h < g; ++h) {
        const size_t row = (size_t)b * Hq + hk * g + h;
        s += expf(logits[row * C + j] - lse[row]);
    }
    float *sc = scores + (size_t)unit * C + j;
    *sc = fmaf(*sc, keep, s * add);
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
    dim3 grid(a.B * a.Hkv, (a.C + 255) / 256);
    k_h2o_decode_acc<<<grid, 256, 0, s>>>(a.Hq, a.Hkv, a.C, a.logits, a.lse, a.n, a.scores, keep,
                                          add, dev_status_ptr());
    return cudaGetLastError();
}

} // namespace kvc
