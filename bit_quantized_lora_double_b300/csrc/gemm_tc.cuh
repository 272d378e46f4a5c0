// gemm_tc.cuh -- definitions shared by the fused NF4-dequant + LoRA GEMM
// (gemm_pair.cuh): the two modes, the launch parameters and the time-bounded
// mbarrier wait.
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

// Stream-K hand-off area, per pair (at most 74): two 512 x 256 fp32
// partial-tile slots (one for the tail of a tile the pair shares with the pairs
// before it, one for the head of a tile it shares with the pairs after it),
// a ready flag per slot, CTA and epilogue warp (16 words), and an arrival
// counter per CTA and epilogue warp for the shared tile the pair heads
// (8 words). All words start at zero.
constexpr int kSkPairs = 74;
constexpr int kSkReadyWords = kSkPairs * 16;
constexpr int kSkFlagWords = kSkPairs * 24;
constexpr int64_t kSlotFloats = 512 * 256;

// Projections of one launch (a group: weights sharing the activation X).
// Forward: the output column tiles of the projections follow one another
// (projection g owns column tiles [cg_first[g], cg_first[g + 1]) of the
// launch), each tile computing Y_g = X W_g'^T + (sU_g) B_g^T. dX: the
// contraction runs over the projections' rows one after another (projection g
// owns main k-steps [kg_first[g], kg_first[g + 1])), so the launch computes
// dX = sum_g dY_g W_g' + (sV) A over all of them.
constexpr int kMaxGroup = 4;

struct TcProj {
    const int8_t *q;
    const float *s2;
    const float *mean;
    const float *absmax;   // per-block fp32 absmax in place of q, s2, mean (null: double-quantized)
    int64_t rows;          // N_g: rows of W_g
    uint16_t *out;         // forward: Y_g; dX: dX (projection 0 only)
    int64_t ldo;
    int64_t ncols;         // valid output columns (forward N_g, dX K)
    int lcol;              // forward: first column of s*U_g in the LoRA activation tensor
    int out_v4;            // out is 16-byte aligned and ldo % 8 == 0: stores through the output tensor map
};

struct TcParams {
    int64_t M;        // rows of the output
    int64_t Nd;       // columns of the launch's output (forward: 256 x column tiles of all projections; dX: K)
    int64_t w_cols;   // K
    int64_t nk_main;  // main k-steps (forward K/64; dX the sum of ceil(N_g/64))
    int lora_steps;   // ceil(r / 64)
    int r;            // width of the LoRA contraction (forward r; dX r x projections)
    int tab;          // level table (kTableNF4 / kTableINT4)
    int ncg;          // column groups: forward the projections, dX 1
    int nkg;          // k groups: dX the projections, forward 1
    int64_t cg_first[kMaxGroup + 1];
    int64_t kg_first[kMaxGroup + 1];
    TcProj pj[kMaxGroup];
    // Stream-K hand-off between pairs (zeroed before the launch):
    // flags [kSkFlagWords] (ready flags, then arrival counters) and two
    // partial-tile slots of kSlotFloats fp32 per pair.
    uint32_t *flags;
    float *slots;
    int64_t dp_tiles;      // tiles t < dp_tiles run data-parallel, the rest stream-K
    int tile_rows;         // rows per tile: 512 (two 256-row sub-tiles) or 256 (one)
    int band;              // row tiles per band of the tile order
    uint64_t wait_ns;
    unsigned kernel_id;
};

// Tensor maps of one launch. Forward: act[0] = X, codes[g], lact = s*U of all
// projections side by side, lw[g] = B_g, out[g] = Y_g. dX: act[g] = dY_g,
// codes[g], lact = s*V of all projections side by side, lw[0] = A of all
// projections stacked, out[0] = dX.
struct GemmMaps {
    CUtensorMap act[kMaxGroup];
    CUtensorMap codes[kMaxGroup];
    CUtensorMap lact;
    CUtensorMap lw[kMaxGroup];
    CUtensorMap out[kMaxGroup];
};

// The k group of main k-step kk.
__host__ __device__ __forceinline__ int kgroup_of(const TcParams &p, int64_t kk) {
    int g = 0;
    while (g + 1 < p.nkg && kk >= p.kg_first[g + 1]) ++g;
    return g;
}

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Limit of the waits that drain a kernel's own asynchronous work (bulk copies
// and tensor-core operations it issued) before it gives up shared memory or
// TMEM. That work always completes, so these waits are independent of the
// adjustable limit of the pipeline waits (which a test may set very low).
constexpr uint64_t kDrainNs = 2000000000ull;

// Waits (at most kDrainNs) for phase `parity` of `bar`; false if it did not
// complete in that time.
__device__ __forceinline__ bool drain_wait(uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer() - t0 > kDrainNs) return false;
    return true;
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


}  // namespace qlora
