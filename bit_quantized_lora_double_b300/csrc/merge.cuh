// merge.cuh -- folds the LoRA adapter into the frozen base weight for
// deployment, before the merged weight is quantized again:
//
//   merged[n, k] = bf16_rne( w'[n, k] + s * t[n, k] ),  t[n, k] = sum_j B[n, j] A[j, k]
//
// Every step is a separately rounded fp32 operation (no fused multiply-add):
// t starts at 0 and adds the products for j = 0 .. r-1 in order (a product
// of two bf16 numbers is exact in fp32), then s * t, then the add to the
// dequantized base weight w' = bf16_rne(L[code] * a'). One thread makes 8
// consecutive weights of a row: 4 code bytes, one absmax code, and for every
// j one element of B and 8 elements of A (a row of A is read by the whole
// row's threads, so it comes from L2).
// Source: xingyuzhitong.com "Fine-Tuning Memory Requirements: Full Training vs
// LoRA vs QLoRA", section "Choosing a method" (adapters are merged into the
// base weights for deployment).
#pragma once

#include "common.cuh"

namespace qlora {

__global__ void __launch_bounds__(256) k_lora_merge(const uint32_t *__restrict__ codes, const int8_t *__restrict__ q,
                                                    const float *__restrict__ s2, const float *__restrict__ mean_p,
                                                    int64_t N, int64_t K, const uint16_t *__restrict__ A,
                                                    const uint16_t *__restrict__ B, int r, float s,
                                                    uint4 *__restrict__ merged) {
    const int64_t chunks = N * K / 8;
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= chunks) return;
    const int64_t n = i / (K / 8), k0 = (i - n * (K / 8)) * 8;
    const int64_t b = (n * K + k0) / kBlock;
    const float a = dq_absmax(__ldg(q + b), __ldg(s2 + (b >> 8)), *mean_p);
    const uint32_t cw = __ldg(codes + i);  // bytes of elements k0 .. k0 + 7, element 2i in the high nibble
    float w[8], t[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const uint32_t byte = (cw >> (8 * (e >> 1))) & 0xFFu;
        const uint32_t code = (e & 1) ? (byte & 15u) : (byte >> 4);
        w[e] = bf16lo_to_f32(__bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(c_levels_q4[kTableNF4][code], a))));
        t[e] = 0.0f;
    }
    for (int j = 0; j < r; ++j) {
        const float bj = bf16lo_to_f32(__ldg(B + n * r + j));
        const uint4 av = __ldg(reinterpret_cast<const uint4 *>(A + (int64_t)j * K + k0));
        const uint32_t as[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            t[2 * e] = __fadd_rn(t[2 * e], __fmul_rn(bj, bf16lo_to_f32(as[e])));
            t[2 * e + 1] = __fadd_rn(t[2 * e + 1], __fmul_rn(bj, bf16hi_to_f32(as[e])));
        }
    }
    uint32_t o[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
        o[e] = pack_bf16x2(__fadd_rn(w[2 * e], __fmul_rn(s, t[2 * e])),
                           __fadd_rn(w[2 * e + 1], __fmul_rn(s, t[2 * e + 1])));
    merged[i] = make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace qlora
