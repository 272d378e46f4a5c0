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
// Dequantize (k_nf4_dequant) reconstructs a' per block, decodes the block's
// 64 codes through the scaled byte-plane table (one block per thread) and
// stages 32 consecutive blocks per warp in shared memory, from where one TMA
// store writes them as 4 KB of contiguous bf16 output.
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

// tab: level table (kTableNF4 / kTableINT4); group_sum may be null (no
// double quantization follows: the absmax values are the stored constants).
__global__ void __launch_bounds__(256) k_nf4_encode(const uint4 *__restrict__ W, int64_t nb,
                                                    uint32_t *__restrict__ codes, float *__restrict__ absmax,
                                                    double *__restrict__ group_sum, int tab) {
    __shared__ float s_thr[16];
    __shared__ float s_abs[kGroup];
    if (threadIdx.x < 15) s_thr[threadIdx.x] = c_thresholds_q4[tab][threadIdx.x];
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
    if (!group_sum) return;
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

constexpr int kDeqWarps = 8;
constexpr int kDeqSmem = kDeqWarps * 2 * 32 * 128 + 1024;  // two 4 KB staging tiles per warp

// One warp per chunk of 32 consecutive blocks (grid-stride over chunks),
// one block per lane: the lane's 32 code bytes (two 16-byte loads, the warp's
// 1 KB contiguous), its int8 absmax code and group scale, the scaled table,
// eight decode8 calls. The 32 x 128-byte rows go to a 128-byte-swizzled
// staging tile (conflict-free 16-byte stores) and one TMA store of the box
// (64 bf16, 32 rows) of the output viewed as [blocks, 64] writes them.
// The next chunk's loads are issued before the current chunk is decoded.
// absmax_f32 (may be null): per-block fp32 absmax used in place of the
// double-quantized q, scale, mean; tab: level table.
__global__ void __launch_bounds__(kDeqWarps * 32) k_nf4_dequant(const __grid_constant__ CUtensorMap tm_out,
                                                               const uint4 *__restrict__ codes,
                                                               const int8_t *__restrict__ q,
                                                               const float *__restrict__ scale,
                                                               const float *__restrict__ mean_p, int64_t nb,
                                                               const float *__restrict__ absmax_f32, int tab) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *stage = smem + warp * 2 * 4096;
    const int64_t nchunks = (nb + 31) / 32;
    const int64_t nw = (int64_t)gridDim.x * kDeqWarps;
    const float mean = absmax_f32 ? 0.0f : *mean_p;
    int64_t c = (int64_t)blockIdx.x * kDeqWarps + warp;
    uint4 cw0 = make_uint4(0, 0, 0, 0), cw1 = cw0;
    int qv = 0;
    float sv = 0.0f;
    auto load = [&](int64_t ch) {
        const int64_t b = ch * 32 + lane;
        if (ch < nchunks && b < nb) {
            cw0 = __ldg(codes + 2 * b);
            cw1 = __ldg(codes + 2 * b + 1);
            if (absmax_f32) {
                sv = __ldg(absmax_f32 + b);
            } else {
                qv = __ldg(q + b);
                sv = __ldg(scale + (b >> 8));
            }
        }
    };
    load(c);
    uint32_t it = 0;
    for (; c < nchunks; c += nw, ++it) {
        const uint32_t w[8] = {cw0.x, cw0.y, cw0.z, cw0.w, cw1.x, cw1.y, cw1.z, cw1.w};
        const Nf4Table tbl = make_table(absmax_f32 ? sv : dq_absmax((int8_t)qv, sv, mean), tab);
        load(c + nw);
        uint8_t *buf = stage + (it & 1) * 4096;
        if (lane == 0) bulk_wait_read<1>();  // the store that last read this tile is done with it
        __syncwarp();
        uint8_t *row = buf + lane * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint32_t o[4];
            decode8(tbl, w[j], o);
            *reinterpret_cast<uint4 *>(row + ((j ^ (lane & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(&tm_out, buf, 0, (int32_t)(c * 32));
            bulk_commit();
        }
    }
    if (lane == 0) bulk_wait_all();
}

}  // namespace qlora
