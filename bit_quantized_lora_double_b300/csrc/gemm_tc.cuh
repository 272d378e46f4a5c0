// gemm_tc.cuh -- definitions shared by the fused NF4-dequant + LoRA GEMM
// (gemm_pair.cuh): the two modes, the launch parameters, the time-bounded
// mbarrier wait and the reduction of contraction-split partials.
//
//   forward (kFwd):  Y [M, N]  = X [M, K]  . W'^T       + (sU) [M, r] . B^T
//   dX      (kDx):   dX [M, K] = dY [M, N] . W'          + (sV) [M, r] . A
//
// Sources: ashishsrivastav.com "QLoRA: Fine-Tuning a 70B on One GPU", section
// "Double Quantization" (dequantize on the fly for the matmul);
// xingyuzhitong.com "Fine-Tuning Memory Requirements", section "QLoRA: quantize
// the frozen base to 4 bits".
#pragma once

#include "common.cuh"

namespace qlora {

enum { kFwd = 0, kDx = 1 };

// Contraction steps are 64 deep (one NF4 block of a weight row).
constexpr int kGemmBK = 64;

struct TcParams {
    int64_t M;        // rows of the output
    int64_t Nd;       // columns of the output (N for forward, K for dX)
    int64_t w_rows;   // N
    int64_t w_cols;   // K
    int64_t nk_main;  // main k-steps (K/64 forward, ceil(N/64) dX)
    int lora_steps;   // ceil(r / 64)
    int r;
    const int8_t *q;
    const float *s2;
    const float *mean;
    uint16_t *out;
    int64_t ldo;
    int splits;            // contraction splits (grid.z); 1 = no split
    int64_t steps_per_split;
    float *part;           // splits > 1: fp32 partials [splits][M][Nd]
    uint64_t wait_ns;
    unsigned kernel_id;
    int out_v8;            // out and ldo allow 32-byte stores of 64-column segments
};

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of `bar` with a time limit; false (and the error
// word recorded) when the limit runs out or another role already aborted.
__device__ __forceinline__ bool tc_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns, unsigned code,
                                        volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 4; ++i)
            if (mbar_try_wait_sleep(bar, parity, kWaitHintNs)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > limit_ns) {
            record_error(code);
            *abort_flag = 1;
            return false;
        }
    }
}

// out[row, col] = bf16( sum over splits, in split order, of part[z][row][col] )
__global__ void k_split_reduce(const float *__restrict__ part, int splits, int64_t M, int64_t Nd,
                               uint16_t *__restrict__ out, int64_t ldo) {
    const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (i >= M * Nd) return;
    const int64_t row = i / Nd, col = i % Nd;
    if (col + 4 <= Nd && (Nd & 3) == 0) {
        float4 a = reinterpret_cast<const float4 *>(part + i)[0];
        for (int zz = 1; zz < splits; ++zz) {
            const float4 b = reinterpret_cast<const float4 *>(part + (int64_t)zz * M * Nd + i)[0];
            a.x += b.x;
            a.y += b.y;
            a.z += b.z;
            a.w += b.w;
        }
        uint2 pk;
        pk.x = pack_bf16x2(a.x, a.y);
        pk.y = pack_bf16x2(a.z, a.w);
        if ((ldo & 3) == 0) {
            *reinterpret_cast<uint2 *>(out + row * ldo + col) = pk;
            return;
        }
        out[row * ldo + col] = (uint16_t)(pk.x & 0xFFFF);
        out[row * ldo + col + 1] = (uint16_t)(pk.x >> 16);
        out[row * ldo + col + 2] = (uint16_t)(pk.y & 0xFFFF);
        out[row * ldo + col + 3] = (uint16_t)(pk.y >> 16);
        return;
    }
    for (int e = 0; e < 4 && i + e < M * Nd; ++e) {
        const int64_t ii = i + e, r = ii / Nd, c = ii % Nd;
        float a = part[ii];
        for (int zz = 1; zz < splits; ++zz) a += part[(int64_t)zz * M * Nd + ii];
        out[r * ldo + c] = __bfloat16_as_ushort(__float2bfloat16_rn(a));
    }
}

}  // namespace qlora
