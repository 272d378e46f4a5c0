// codec.cuh -- NF4 quantizer (encode, double quantization) and dequantizer.
//
// Quantize runs three kernels:
//   k_nf4_encode      one CTA per group of 256 blocks: loads 8 bf16 per thread
//                     (16 B, coalesced), block absmax over 8 lanes, fp32
//                     x = w / absmax, nearest level by a 4-step search over the
//                     15 midpoint thresholds, packs 8 codes into one 32-bit
//                     word; then a pairwise fp64 tree over the group's 256
//                     absmax values.
//   k_pairwise_reduce continues the same tree over the group sums, 256 at a
//                     time, until one value is left: S; mean = fp32(S / nb).
//   k_dq_encode       one warp per group: c = a - mean, scale = max|c| / 127,
//                     q = rint(c / scale) clamped to [-127, 127].
// Dequantize (k_nf4_dequant) reconstructs a' per block and decodes 32 codes
// per thread through the scaled byte-plane table.
// Sources: ashishsrivastav.com "QLoRA: Fine-Tuning a 70B on One GPU", sections
// "NF4 Quantization: Beyond Standard INT4" and "Double Quantization: Squeezing
// the Constants"; inquiringlines.com note, mechanism paragraph.
#pragma once

#include "common.cuh"

namespace qlora {

// Pairwise sum of 8 values held by one thread: ((0+1)+(2+3))+((4+5)+(6+7)).
__device__ __forceinline__ double tree8(const double (&v)[8]) {
    return ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
}

// Warp-wide continuation of the tree: xor-shuffles 1, 2, 4, 8, 16 add
// neighbouring subtrees (addition is commutative, so both partners hold the
// same value at every level). Lane 0 ends with the 256-leaf tree.
__device__ __forceinline__ double tree_warp(double v) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) v = v + __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Nearest NF4 code of an fp32 x in [-1, 1] (number of thresholds strictly
// below x), by binary search over the 15 thresholds held in shared memory.
__device__ __forceinline__ uint32_t nf4_code(float x, const float *thr) {
    uint32_t c = (x > thr[7]) ? 8u : 0u;
    c += (x > thr[c + 3]) ? 4u : 0u;
    c += (x > thr[c + 1]) ? 2u : 0u;
    c += (x > thr[c]) ? 1u : 0u;
    return c;
}

__global__ void __launch_bounds__(256) k_nf4_encode(const uint4 *__restrict__ W, int64_t nb,
                                                    uint32_t *__restrict__ codes, float *__restrict__ absmax,
                                                    double *__restrict__ group_sum) {
    __shared__ float s_thr[16];
    __shared__ float s_abs[kGroup];
    if (threadIdx.x < 15) s_thr[threadIdx.x] = c_thresholds[threadIdx.x];
    __syncthreads();
    const int64_t g = blockIdx.x;
    const int sub = threadIdx.x & 7;   // which 8-element slice of the block
    const int lb0 = threadIdx.x >> 3;  // block within a pass of 32 blocks
#pragma unroll 1
    for (int pass = 0; pass < kGroup / 32; ++pass) {
        const int lb = pass * 32 + lb0;
        const int64_t b = g * kGroup + lb;
        const bool valid = b < nb;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (valid) v = W[b * 8 + sub];
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
        float f[8];
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = bf16lo_to_f32(wv[i]);
            f[2 * i + 1] = bf16hi_to_f32(wv[i]);
            m = fmaxf(m, fmaxf(fabsf(f[2 * i]), fabsf(f[2 * i + 1])));
        }
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
        if (sub == 0) {
            s_abs[lb] = valid ? m : 0.0f;
            if (valid) absmax[b] = m;
        }
        if (valid) {
            uint32_t word = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t c0 = 7u, c1 = 7u;
                if (m != 0.0f) {
                    c0 = nf4_code(__fdiv_rn(f[2 * j], m), s_thr);
                    c1 = nf4_code(__fdiv_rn(f[2 * j + 1], m), s_thr);
                }
                word |= ((c0 << 4) | c1) << (8 * j);
            }
            codes[b * 8 + sub] = word;
        }
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        double v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = static_cast<double>(s_abs[threadIdx.x * 8 + i]);
        double s = tree_warp(tree8(v));
        if (threadIdx.x == 0) group_sum[g] = s;
    }
}

// One warp per chunk of 256 inputs (zero-padded): out[chunk] = tree sum.
// When `mean_out` is set (last level, n <= 256), writes fp32(S / nb).
__global__ void __launch_bounds__(256) k_pairwise_reduce(const double *__restrict__ in, int64_t n,
                                                         double *__restrict__ out, float *__restrict__ mean_out,
                                                         int64_t nb) {
    const int64_t chunk = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (chunk > 0 && chunk * 256 >= n) return;  // chunk 0 always runs (n <= 256 at the last level)
    double v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t idx = chunk * 256 + lane * 8 + i;
        v[i] = idx < n ? in[idx] : 0.0;
    }
    const double s = tree_warp(tree8(v));
    if (lane == 0) {
        if (mean_out) {
            *mean_out = static_cast<float>(s / static_cast<double>(nb));
        } else {
            out[chunk] = s;
        }
    }
}

__global__ void __launch_bounds__(256) k_dq_encode(const float *__restrict__ absmax, int64_t nb,
                                                   const float *__restrict__ mean_p, int8_t *__restrict__ q,
                                                   float *__restrict__ scale) {
    const int64_t g = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int64_t ng = (nb + kGroup - 1) / kGroup;
    if (g >= ng) return;
    const float mean = *mean_p;
    float c[8];
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t b = g * kGroup + lane * 8 + i;
        c[i] = b < nb ? __fsub_rn(absmax[b], mean) : 0.0f;
        m = fmaxf(m, fabsf(c[i]));
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float s2 = __fdiv_rn(m, 127.0f);
    if (lane == 0) scale[g] = s2;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t b = g * kGroup + lane * 8 + i;
        if (b < nb) {
            int v = 0;
            if (s2 != 0.0f) {
                v = __float2int_rn(__fdiv_rn(c[i], s2));
                v = v > 127 ? 127 : (v < -127 ? -127 : v);
            }
            q[b] = static_cast<int8_t>(v);
        }
    }
}

// Each thread decodes 32 codes (16 bytes = half of one block) into 64 bytes
// of bf16.
__global__ void __launch_bounds__(256) k_nf4_dequant(const uint4 *__restrict__ codes,
                                                     const int8_t *__restrict__ q,
                                                     const float *__restrict__ scale,
                                                     const float *__restrict__ mean_p, int64_t nhalf,
                                                     uint4 *__restrict__ out) {
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= nhalf) return;
    const int64_t b = t >> 1;
    const float a = dq_absmax(q[b], scale[b / kGroup], *mean_p);
    const Nf4Table tab = make_table(a);
    const uint4 cw = codes[t];
    const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t o[4];
        decode8(tab, w[i], o);
        out[t * 4 + i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

}  // namespace qlora
