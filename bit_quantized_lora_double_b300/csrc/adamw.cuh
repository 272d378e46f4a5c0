// adamw.cuh -- one AdamW step for the LoRA adapters, with the optimizer
// state (and the fp32 master weights) wherever the caller keeps them: device
// memory, managed memory that the driver pages between host and device, or
// pinned host memory read over the interconnect ("paged optimizers").
//
//   p = p * decay                       decay = 1 - lr * wd   (decoupled weight decay)
//   m = b1 m + (1 - b1) g ;  v = b2 v + (1 - b2) g^2
//   p = p - step * m / (sqrt(v) / c2 + eps)    step = lr / (1 - b1^t), c2 = sqrt(1 - b2^t)
//
// and, when asked, the bf16 copy of p that the next forward pass reads.
// Four parameters per thread and iteration (16-byte accesses), grid-stride.
// Sources: inquiringlines.com note, mechanism paragraph (paged optimizers);
// ashishsrivastav.com "QLoRA: Fine-Tuning a 70B on One GPU", section "Paged
// Optimizers: Managing Fragmentation"; the AdamW rule itself is the usual
// decoupled-decay form, which the pages name (paged_adamw) but do not spell out.
#pragma once

#include "common.cuh"

namespace qlora {

struct AdamwParams {
    float decay, b1, b2, one_m_b1, one_m_b2, step, c2, eps;
};

__device__ __forceinline__ float adamw_one(float &p, float g, float &m, float &v, const AdamwParams &h) {
    p = p * h.decay;
    m = fmaf(h.b1, m, h.one_m_b1 * g);
    v = fmaf(h.b2, v, h.one_m_b2 * g * g);
    p = p - h.step * m / (sqrtf(v) / h.c2 + h.eps);
    return p;
}

__global__ void __launch_bounds__(256) k_adamw(float *__restrict__ p, uint16_t *__restrict__ pb,
                                               const float *__restrict__ g, float *__restrict__ m,
                                               float *__restrict__ v, int64_t n, AdamwParams h) {
    const int64_t n4 = n / 4;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
        float4 pp = reinterpret_cast<float4 *>(p)[i], mm = reinterpret_cast<float4 *>(m)[i],
               vv = reinterpret_cast<float4 *>(v)[i];
        const float4 gg = reinterpret_cast<const float4 *>(g)[i];
        adamw_one(pp.x, gg.x, mm.x, vv.x, h);
        adamw_one(pp.y, gg.y, mm.y, vv.y, h);
        adamw_one(pp.z, gg.z, mm.z, vv.z, h);
        adamw_one(pp.w, gg.w, mm.w, vv.w, h);
        reinterpret_cast<float4 *>(p)[i] = pp;
        reinterpret_cast<float4 *>(m)[i] = mm;
        reinterpret_cast<float4 *>(v)[i] = vv;
        if (pb) reinterpret_cast<uint2 *>(pb)[i] = make_uint2(pack_bf16x2(pp.x, pp.y), pack_bf16x2(pp.z, pp.w));
    }
    // the last n % 4 parameters
    for (int64_t i = n4 * 4 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        float pp = p[i], mm = m[i], vv = v[i];
        adamw_one(pp, g[i], mm, vv, h);
        p[i] = pp;
        m[i] = mm;
        v[i] = vv;
        if (pb) pb[i] = __bfloat16_as_ushort(__float2bfloat16_rn(pp));
    }
}

}  // namespace qlora
