// fwd_few.cuh -- forward of the NF4 LoRA linear layer for a few tokens
// (M <= 16, decode-like), bound by streaming the packed weight from HBM.
//
//   Y [M, N] = X [M, K] . W'^T + (sU) [M, r] . B^T          (K % 256 == 0)
//
// One launch serves one projection or a group of up to four sharing X and K
// (their row tiles one after the other in a single line of tiles, each with
// its own tensor map, constants, B, Y and slice of sU).
//
// Work: the weight is cut into tasks of 32 rows x 256 k (four blocks of 64;
// the codes of a task are one TMA box of 32 rows x 128 bytes), numbered row
// tile by row tile: tile t holds tasks [t P, (t + 1) P), P = K / 256. The
// line of T tasks is split evenly over the W warps of the grid (16 warps a
// CTA with one 8-token tile, 12 with two; warp w = warps a CTA * block +
// warp index takes [w T / W, (w + 1) T / W), at least one task each), so the
// SMs stream the same number of bytes to within a task.
//
// Every warp is its own pipeline: its lane 0 keeps two of its tasks in flight
// (two 4 KB slots, one mbarrier each), the warp decodes a landed task while
// the next one streams, and refills the slot it just read. After the start no
// barrier couples the warps of a CTA.
//
// Decode: entry b of the byte table in shared memory holds the bf16 pair
// (L[b >> 4], L[b & 15]) of the two codes a byte b packs, one copy per lane
// (a warp's 32 lookups hit 32 banks) at a stride of 256 bytes; the table sits
// at a 64 KB-aligned shared address, so one PRMT merges a code byte into the
// lane's base to form the lookup address. The pairs are the A fragments of
// mma.sync m16n8k16 (two 16-row tiles), multiplied with X^T fragments (k
// permuted identically in A and X inside each block); each block's fp32 sum
// is scaled by the block's reconstructed absmax a' = fp32(q) * scale + mean,
// so a weight enters as bf16(L[code]) * a' (within one bf16 rounding of
// bf16(L[code] * a')).
//
// A row tile is finished when a warp's range leaves it. A tile inside one
// warp's range: that warp adds the LoRA term sU . B^T (one more mma.sync per
// 16 ranks) and writes the outputs as bf16. A tile shared by several warps:
// each writes its fp32 fragments to its slot in the workspace and bumps the
// tile's arrival counter; the warp that arrives last adds all the slots in
// warp order and finishes the tile. Nothing waits on another warp.
// Sources: ashishsrivastav.com "QLoRA: Fine-Tuning a 70B on One GPU", section
// "Double Quantization" (dequantize on the fly); xingyuzhitong.com
// "Fine-Tuning Memory Requirements", section "QLoRA: quantize the frozen base
// to 4 bits".
#pragma once

#include "common.cuh"
#include "gemm_tc.cuh"
#include "small_m.cuh"

namespace qlora {

struct FewCfg {
    static constexpr int ROWS = 32;                     // weight rows per task (two m16 tiles)
    static constexpr int TK = 256;                      // k per task: four blocks
    static constexpr int WARPS = 16;                    // warps per CTA at most, one pipeline each
    static constexpr int THREADS = 32 * WARPS;
    static constexpr int TASK_BYTES = ROWS * 128;       // a task's codes: one 32-row x 128-byte box
    static constexpr int SLOTS = 2;                     // tasks in flight per warp
    static constexpr int NSLOT = WARPS * SLOTS;
    static constexpr int NBAR = WARPS * SLOTS;
    static constexpr int MAX_NT = 2;                    // 8-token tiles: up to 16 tokens
    static constexpr uint32_t TABLE_ADDR = 0x10000;     // shared address of the byte table (64 KB aligned)
    static constexpr uint32_t TABLE_BYTES = 0x10000;    // 256 entries x 256 bytes (lane copies in the first 128)
    // Dynamic shared memory: ring slots below the table (from the first
    // 1024-byte boundary of the allocation) and above it, then the barriers.
    // Covers any allocation start up to 4 KB into the shared window (the
    // kernel checks its layout and records an error otherwise).
    static constexpr int SMEM_BYTES = 200704;
    static constexpr int GRID = 148;                    // CTAs at most (one per SM)
};
static_assert(FewCfg::TASK_BYTES % 1024 == 0, "128-byte swizzle alignment of the slots");
static_assert(FewCfg::TABLE_ADDR + FewCfg::TABLE_BYTES + (FewCfg::NSLOT - 15) * FewCfg::TASK_BYTES +
                      FewCfg::NBAR * 8 + 16 <=
                  0x400 + FewCfg::SMEM_BYTES,
              "layout when the allocation starts 1 KB into the window (15 slots below the table)");
static_assert(FewCfg::SMEM_BYTES <= 232448, "shared memory per CTA");

// Warps per CTA for NT 8-token tiles: sixteen with one tile; twelve with two
// (their accumulators and the X fragments requested a block ahead need the
// registers of a 384-thread CTA).
template <int NT>
__host__ __device__ constexpr int few_warps() {
    return NT == 1 ? 16 : 12;
}
static_assert(few_warps<1>() <= FewCfg::WARPS && few_warps<2>() <= FewCfg::WARPS, "slots of the layout");

// Diagnostic timeline (built only with -DQLORA_GEMM_STAMPS, into a separate
// library): globaltimer stamps per warp of the last launch. Columns: 0 entry,
// 1 after the start barrier, 2 + 2 i / 3 + 2 i task i landed / decoded (i < 4),
// 10 / 11 and 12 / 13 first and second tile end begun / done, 14 stream done,
// 15 tiles this warp finished.
#ifdef QLORA_GEMM_STAMPS
constexpr int kFewStampWarps = FewCfg::WARPS * FewCfg::GRID;
__device__ unsigned long long d_few_stamps[kFewStampWarps][16];
#define QLORA_FEW_STAMP(w, col) \
    do {                        \
        if (lane == 0) d_few_stamps[w][col] = globaltimer(); \
    } while (0)
#else
#define QLORA_FEW_STAMP(w, col) \
    do {                        \
    } while (0)
#endif

// One projection of a launch (up to kMaxGroup projections that share X and
// K): its weight's constants, its adapter's B and its output, and where its
// row tiles start in the launch's line of tiles.
struct FewProj {
    const int8_t *q;       // int8 absmax codes [N, K / 64] (null with fp32 absmax)
    const float *s2;       // second-level scales, one per 256 blocks
    const float *mean;
    const float *absmax;   // fp32 block absmax (variant without double quantization)
    const uint16_t *B;     // [N, r]
    uint16_t *Y;           // [M, N]
    int64_t N;
    uint32_t tile0;        // first row tile of this projection in the launch
    int sucol;             // first column of its bf16(s * U) slice in sU
};
// NP: projections a launch carries room for (1, or kMaxGroup for groups), so
// that a single projection's kernel parameters stay small.
template <int NP>
struct FewMaps {
    CUtensorMap codes[NP];  // the packed codes of each projection
};
template <int NP>
struct FewParams {
    const uint16_t *X;
    int64_t M, K;
    const uint16_t *sU;    // bf16(s * U) [M, ldu]: one slice of 64-column multiples per projection, zero beyond r
    int ldu;
    int r;
    int nproj;
    FewProj proj[NP];
    float *slots;          // [warps][2][32 lanes][8 NT]: fragments of shared row tiles
    uint32_t *counters;    // [row tiles of all projections], zeroed by the preceding kernel
    int64_t tasks;         // T = row tiles x P
    int64_t tpr;           // P = K / 256 tasks per row tile
    int64_t warps;         // W = min(T, warps a CTA x grid)
    uint64_t wait_ns;
    float levels[16];      // the 4-bit level table (a kernel parameter: no cold constant-cache read)
};

// first task of warp w of W (T < 2^31 tasks, W < 2^16 warps; 32-bit
// division whenever w * T fits in 32 bits: every realistic shape)
__host__ __device__ __forceinline__ uint32_t few_begin(uint32_t w, uint32_t W, uint32_t T) {
    const uint64_t x = (uint64_t)w * T;
    return x < (uint64_t(1) << 32) ? (uint32_t)x / W : (uint32_t)(x / W);
}

// the warp whose range holds task x (T >= W: no range is empty)
__host__ __device__ __forceinline__ uint32_t few_owner(uint32_t x, uint32_t W, uint32_t T) {
    const uint64_t y = (uint64_t)(x + 1) * W - 1;
    return y < (uint64_t(1) << 32) ? (uint32_t)y / T : (uint32_t)(y / T);
}

// Shared-memory layout of one launch (shared-window addresses): slot i at
// lo + 4096 i for i < nlo, else at hi + 4096 (i - nlo); barriers at bars.
struct FewLayout {
    uint32_t lo, nlo, hi, bars;
};
__device__ __forceinline__ bool few_layout(uint32_t base, FewLayout &L) {
    using C = FewCfg;
    L.lo = (base + 1023u) & ~1023u;
    L.nlo = L.lo <= C::TABLE_ADDR ? (C::TABLE_ADDR - L.lo) / C::TASK_BYTES : 0u;
    if (L.nlo > (uint32_t)C::NSLOT) L.nlo = C::NSLOT;
    L.hi = C::TABLE_ADDR + C::TABLE_BYTES;
    L.bars = L.hi + ((uint32_t)C::NSLOT - L.nlo) * C::TASK_BYTES;
    return base <= C::TABLE_ADDR && L.bars + C::NBAR * 8 + 16 <= base + (uint32_t)C::SMEM_BYTES;
}
__device__ __forceinline__ uint32_t few_slot(const FewLayout &L, int i) {
    return (uint32_t)i < L.nlo ? L.lo + (uint32_t)i * FewCfg::TASK_BYTES
                               : L.hi + ((uint32_t)i - L.nlo) * FewCfg::TASK_BYTES;
}

// One table lookup: byte J of w, merged into the lane's table address
// (TABLE_ADDR | 4 * lane: bytes 0 and 2 kept, byte 1 replaced).
template <int J>
__device__ __forceinline__ uint32_t few_lut(uint32_t w, uint32_t lanebase) {
    uint32_t a, v;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(a) : "r"(w), "r"(lanebase), "n"(0x7604 | (J << 4)));
    asm("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// arrival on a row tile's counter: release of this warp's slot stores,
// acquire of the other contributors' (whoever arrives last reads them)
__device__ __forceinline__ uint32_t few_atom_add_acq_rel(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// D = A * B (+ D): mma.sync without side effects, so that the compiler may
// interleave it with the table lookups
__device__ __forceinline__ void few_mma_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %10, %10, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}
__device__ __forceinline__ void few_mma(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// sU for the few-token forward over n projections (A_g [r, K] each): CTA
// (m, jj, g) computes U[m, j] = sum_k X[m, k] A_g[jj, k], j = g r + jj (threads
// striding over K in 8-element chunks, eight loads of each operand in
// flight, then a warp and a block reduction in fixed order) and writes U
// (bf16, stride ldu, may be null) and sU = bf16(s * U) at column g rp + jj
// (stride lds: one slice of rp columns per projection); CTA (m, 0, g) also
// writes the zeros of slice g beyond r, and CTA (0, 0) zeroes the forward's
// arrival counters. A0..A3: A_g (unused ones may be null). K % 8 == 0.
// Grid: (M, r, n).
constexpr int kFewDownThreads = 256;
__global__ void __launch_bounds__(kFewDownThreads) k_few_down(const uint16_t *__restrict__ X, int64_t K,
                                                              const uint16_t *__restrict__ A0,
                                                              const uint16_t *__restrict__ A1,
                                                              const uint16_t *__restrict__ A2,
                                                              const uint16_t *__restrict__ A3, int r, float s,
                                                              uint16_t *__restrict__ U, int ldu,
                                                              uint16_t *__restrict__ sU, int lds, int rp,
                                                              uint32_t *__restrict__ zero, int nzero) {
    // launched as a programmatic dependent of whatever precedes it: wait for
    // that grid before touching memory (X or the workspace may be its output)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the forward, launched as a programmatic dependent, may start streaming
    // its weights now; it waits for this grid before it reads sU or counts
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ float wsum[kFewDownThreads / 32];
    const int m = blockIdx.x, jj = blockIdx.y, pj = blockIdx.z, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j = pj * r + jj;
    if (m == 0 && j == 0)
        for (int i = threadIdx.x; i < nzero; i += kFewDownThreads) zero[i] = 0u;
    if (jj == 0)  // the zero columns of this projection's slice
        for (int i = r + threadIdx.x; i < rp; i += kFewDownThreads) sU[(int64_t)m * lds + pj * rp + i] = 0;
    const uint16_t *Ap = pj == 0 ? A0 : (pj == 1 ? A1 : (pj == 2 ? A2 : A3));
    const uint4 *xr = reinterpret_cast<const uint4 *>(X + (int64_t)m * K);
    const uint4 *ar = reinterpret_cast<const uint4 *>(Ap + (int64_t)jj * K);
    float acc = 0.0f;
#pragma unroll 8
    for (int64_t c = threadIdx.x; c < K / 8; c += kFewDownThreads) {
        const uint4 x = __ldg(xr + c), a = __ldg(ar + c);
        const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, as[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            acc = fmaf(bf16lo_to_f32(xs[e]), bf16lo_to_f32(as[e]), acc);
            acc = fmaf(bf16hi_to_f32(xs[e]), bf16hi_to_f32(as[e]), acc);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) wsum[warp] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = wsum[0];
#pragma unroll
        for (int w = 1; w < kFewDownThreads / 32; ++w) t += wsum[w];
        if (U) U[(int64_t)m * ldu + j] = __bfloat16_as_ushort(__float2bfloat16_rn(t));
        sU[(int64_t)m * lds + pj * rp + jj] = __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(s, t)));
    }
}

// NT = number of 8-token tiles (M <= 8 * NT <= 16).
// F32A: the block absmax is stored as fp32 (`absmax`, one per block) instead
// of double-quantized; the level table comes in p.levels.
// MULTI: more than one projection (p.nproj > 1); with one, every projection
// lookup folds to projection 0.
template <int NT, bool F32A, bool MULTI>
__global__ void __launch_bounds__(32 * few_warps<NT>(), 1)
    k_fwd_few(const __grid_constant__ FewMaps<MULTI ? kMaxGroup : 1> tm,
              const __grid_constant__ FewParams<MULTI ? kMaxGroup : 1> p) {
    using C = FewCfg;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = smem_u32(smem_raw);
    FewLayout L;
    if (!few_layout(base, L)) {
        if (threadIdx.x == 0) record_error((10u << 16) | 9u);
        return;
    }
    auto sp = [&](uint32_t a) { return smem_raw + (a - base); };
    // the next kernel, if launched as a programmatic dependent, may be
    // scheduled now (it waits for this grid before touching memory)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t T = (uint32_t)p.tasks, W = (uint32_t)p.warps, P = (uint32_t)p.tpr;
    constexpr int WPC = few_warps<NT>();  // warps of this CTA
    const uint32_t gw = blockIdx.x * WPC + warp;
    const bool active = gw < W;
    if (active) QLORA_FEW_STAMP(gw, 0);
    const uint32_t t0 = active ? few_begin(gw, W, T) : 0, t1 = active ? few_begin(gw + 1, W, T) : 0;
    const int n = (int)(t1 - t0);
    uint64_t *full = reinterpret_cast<uint64_t *>(sp(L.bars)) + C::SLOTS * warp;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sp(L.bars + C::NBAR * 8));
    constexpr int S = C::SLOTS;  // this warp's slots
    // this warp's slot s (1024-byte aligned; the table may sit between two)
    auto slot_of = [&](int s) { return few_slot(L, C::SLOTS * warp + s); };

    // the projection whose row tiles hold the launch's tile gt
    auto proj_of = [&](uint32_t gt) {
        int pj = 0;
#pragma unroll
        for (int k = 1; k < (MULTI ? kMaxGroup : 1); ++k) pj += (k < p.nproj && gt >= p.proj[k].tile0) ? 1 : 0;
        return pj;
    };
    // lane 0: task x into slot s (tile x / P: rows 32 (tile - its
    // projection's first) .., bytes 128 (x % P) .. of that projection's codes)
    auto issue = [&](int s, uint32_t x) {
        const uint32_t gt = x / P, kc = x - gt * P;
        const int pj = proj_of(gt);
        mbar_arrive_expect_tx(&full[s], (uint32_t)C::TASK_BYTES);
        tma_load_2d(sp(slot_of(s)), &tm.codes[pj], &full[s], (int32_t)(kc * 128u),
                    (int32_t)((gt - p.proj[pj].tile0) * C::ROWS));
    };
    if (threadIdx.x == 0) *abort_flag = 0;
    if (lane == 0 && active) {
        for (int k = 0; k < p.nproj; ++k) prefetch_tmap(&tm.codes[k]);
        for (int q = 0; q < S; ++q) mbar_init(&full[q], 1);
        fence_mbar_init();
        fence_proxy_async_smem();
        for (int q = 0; q < S && q < n; ++q) issue(q, t0 + q);
    }
    // the byte table, while the first tasks stream in: word (e, lane) at
    // TABLE_ADDR + 256 e + 4 lane = bf16 pair (L[e >> 4] low, L[e & 15] high)
    for (int i = threadIdx.x; i < 256 * 32; i += 32 * WPC) {
        const int e = i >> 5, l = i & 31;
        *reinterpret_cast<uint32_t *>(sp(C::TABLE_ADDR + (uint32_t)(e * 256 + l * 4))) =
            pack_bf16x2(p.levels[e >> 4], p.levels[e & 15]);
    }
    __syncthreads();
    if (!active) return;
    QLORA_FEW_STAMP(gw, 1);
    int n_end = 0, n_fin = 0;

    const int g = lane >> 2, t = lane & 3;
    const uint32_t lanebase = C::TABLE_ADDR | (uint32_t)(lane << 2);
    const uint32_t KB = (uint32_t)(p.K / kBlock);
    const float mean0 = F32A ? 0.0f : __ldg(p.proj[0].mean);  // (one projection)
    // X^T fragments: token 8 j + g, k = 64 kb + 16 t .. + 15
    const uint16_t *xb[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) xb[j] = 8 * j + g < p.M ? p.X + (8 * j + g) * p.K + 16 * t : nullptr;
    // this lane's 8 code bytes of row g + 8 q, block b in a slot (128-byte
    // rows, 128-byte swizzle: 16-byte chunk h of row r sits at h ^ (r & 7))
    auto code_off = [&](int q, int b) {
        return (uint32_t)(g * 128 + 1024 * q + ((((2 * b + (t >> 1)) ^ g)) << 4) + (t & 1) * 8);
    };

    // Block scales of a task for rows g + 8 i (i < 4) and its four blocks:
    // the int8 codes as one word per row (blocks 4 kc .. 4 kc + 3, all in one
    // group of 256) and the row's second-level scale, or the fp32 absmax.
    // Rows past the last one read row 0: their outputs are never written.
    struct Scales {
        uint32_t q[4];
        float s2[4];
        float4 a[4];
        float mean;
    };
    auto load_scales = [&](uint32_t x, Scales &sc) {
        const uint32_t gt = x / P, kc = x - gt * P;
        // (the parameters are read by index, never through a reference: a
        // constant-bank load, folded to an immediate with one projection)
        const int pj = proj_of(gt);
        const uint32_t row0 = (gt - p.proj[pj].tile0) * C::ROWS;
        if (MULTI && !F32A) sc.mean = __ldg(p.proj[pj].mean);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t nrow = row0 + g + 8 * i;
            const uint32_t idx = (nrow < (uint32_t)p.proj[pj].N ? nrow : 0u) * KB + 4u * kc;
            if (F32A) {
                sc.a[i] = __ldg(reinterpret_cast<const float4 *>(p.proj[pj].absmax + idx));
            } else {
                sc.q[i] = __ldg(reinterpret_cast<const uint32_t *>(p.proj[pj].q + idx));
                sc.s2[i] = __ldg(p.proj[pj].s2 + (idx >> 8));
            }
        }
    };

    bool pdl_done = false;
    auto pdl_wait_once = [&]() {
        // sU and the zeroed counters come from the preceding kernel (launched
        // before this one as a programmatic dependency)
        if (!pdl_done) {
            asm volatile("griddepcontrol.wait;" ::: "memory");
            pdl_done = true;
        }
    };
    // B pair (B[n, jj], B[n, jj + 1]) of projection pr as bf16x2, zero
    // beyond its N rows or r ranks
    auto b_pair = [&](int pj, int64_t nrow, int jj) -> uint32_t {
        if (nrow >= p.proj[pj].N || jj >= p.r) return 0u;
        const uint16_t *br = p.proj[pj].B + nrow * p.r + jj;
        if ((p.r & 1) == 0) return __ldg(reinterpret_cast<const uint32_t *>(br));  // 4-byte aligned
        const uint32_t hi = jj + 1 < p.r ? (uint32_t)__ldg(br + 1) : 0u;
        return (uint32_t)__ldg(br) | (hi << 16);
    };
    // LoRA operands of ranks [16 kk, 16 kk + 16) for the projection's row
    // tile lt: rows of B as A fragments, sU^T as B fragments (its slice of sU
    // is zero beyond r)
    auto lora_a = [&](int pj, uint32_t lt, int kk, uint32_t (&ba)[2][4]) {
#pragma unroll
        for (int rt = 0; rt < 2; ++rt) {
            const int64_t ra = (int64_t)lt * C::ROWS + 16 * rt + g;
            ba[rt][0] = b_pair(pj, ra, 16 * kk + 2 * t);
            ba[rt][1] = b_pair(pj, ra + 8, 16 * kk + 2 * t);
            ba[rt][2] = b_pair(pj, ra, 16 * kk + 2 * t + 8);
            ba[rt][3] = b_pair(pj, ra + 8, 16 * kk + 2 * t + 8);
        }
    };
    auto lora_b = [&](int pj, int kk, uint32_t (&bu)[NT][2]) {
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const int tok = 8 * j + g;
            if (tok < p.M) {
                // written by the preceding kernel: read through L2
                const uint16_t *ur = p.sU + (int64_t)tok * p.ldu + p.proj[pj].sucol + 16 * kk + 2 * t;
                bu[j][0] = __ldcg(reinterpret_cast<const unsigned int *>(ur));
                bu[j][1] = __ldcg(reinterpret_cast<const unsigned int *>(ur + 8));
            } else {
                bu[j][0] = bu[j][1] = 0u;
            }
        }
    };
    // Finishes row tile rtile from its full fp32 sums v (fragment layout):
    // adds the LoRA term with mma.sync (ranks 0..15 from ba0 / bu0, loaded
    // by the caller) and writes the valid outputs as bf16.
    auto finish = [&](float (&v)[2][NT][4], int pj, uint32_t lt, const uint32_t (&ba0)[2][4],
                      const uint32_t (&bu0)[NT][2]) {
#pragma unroll
        for (int rt = 0; rt < 2; ++rt)
#pragma unroll
            for (int j = 0; j < NT; ++j) few_mma(v[rt][j], ba0[rt], bu0[j][0], bu0[j][1]);
        for (int kk = 1; kk * 16 < p.r; ++kk) {
            uint32_t ba[2][4], bu[NT][2];
            lora_a(pj, lt, kk, ba);
            lora_b(pj, kk, bu);
#pragma unroll
            for (int rt = 0; rt < 2; ++rt)
#pragma unroll
                for (int j = 0; j < NT; ++j) few_mma(v[rt][j], ba[rt], bu[j][0], bu[j][1]);
        }
        const int64_t row0 = (int64_t)lt * C::ROWS;
#pragma unroll
        for (int rt = 0; rt < 2; ++rt)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t nrow = row0 + 16 * rt + 8 * h + g;
                if (nrow >= p.proj[pj].N) continue;
#pragma unroll
                for (int j = 0; j < NT; ++j)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int tok = 8 * j + 2 * t + e;
                        if (tok < p.M)
                            p.proj[pj].Y[(int64_t)tok * p.proj[pj].N + nrow] =
                                __bfloat16_as_ushort(__float2bfloat16_rn(v[rt][j][2 * h + e]));
                    }
            }
    };

    float acc[2][NT][4];
    auto zero_acc = [&]() {
#pragma unroll
        for (int rt = 0; rt < 2; ++rt)
#pragma unroll
            for (int j = 0; j < NT; ++j) acc[rt][j][0] = acc[rt][j][1] = acc[rt][j][2] = acc[rt][j][3] = 0.0f;
    };
    // Called when this warp's range leaves row tile rtile (tasks [a, a + P)).
    const uint32_t rt_first = t0 / P;
    auto end_tile = [&](uint32_t rtile) {
        if (n_end < 2) QLORA_FEW_STAMP(gw, 10 + 2 * n_end);
        // the first 16 ranks of the LoRA term come in while the tile is
        // handed over (B is an input; sU and the zeroed counters come from
        // the preceding kernel)
        const int pj = proj_of(rtile);
        const uint32_t lt = rtile - p.proj[pj].tile0;
        uint32_t ba0[2][4], bu0[NT][2];
        lora_a(pj, lt, 0, ba0);
        pdl_wait_once();
        lora_b(pj, 0, bu0);
        const uint32_t a = rtile * P, b = a + P;
        if (a >= t0 && b <= t1) {
            finish(acc, pj, lt, ba0, bu0);
            ++n_fin;
            return;
        }
        // shared: this warp's fragments to its slot (0: its first tile, 1: its last)
        const int e = rtile == rt_first ? 0 : 1;
        float4 *mine = reinterpret_cast<float4 *>(p.slots) + ((size_t)(gw * 2 + e) * 32 + lane) * (2 * NT);
#pragma unroll
        for (int rt = 0; rt < 2; ++rt)
#pragma unroll
            for (int j = 0; j < NT; ++j)
                __stcg(mine + rt * NT + j, make_float4(acc[rt][j][0], acc[rt][j][1], acc[rt][j][2], acc[rt][j][3]));
        // the warp barrier orders every lane's stores before lane 0's
        // release (and its acquire before every lane's loads below)
        __syncwarp();
        uint32_t old = 0;
        if (lane == 0) old = few_atom_add_acq_rel(p.counters + rtile, 1u);
        old = __shfl_sync(0xffffffffu, old, 0);
        __syncwarp();
        const uint32_t wa = few_owner(a, W, T), wb = few_owner(b - 1, W, T);
        if (old != (uint32_t)(wb - wa)) return;
        // last to arrive: every contributor's slot. The first contributor's
        // range may start before the tile (then the tile is its last: slot
        // 1); every later one starts inside it (slot 0). Loads of a chunk
        // of contributors are in flight together; the sum runs in warp order.
        ++n_fin;
        const int ea = few_begin(wa, W, T) == a ? 0 : 1;
        constexpr int CH = 4 / NT;
        float v[2][NT][4];
#pragma unroll
        for (int rt = 0; rt < 2; ++rt)
#pragma unroll
            for (int j = 0; j < NT; ++j) v[rt][j][0] = v[rt][j][1] = v[rt][j][2] = v[rt][j][3] = 0.0f;
        for (uint32_t w0 = wa; w0 <= wb; w0 += CH) {
            float4 u[CH][2 * NT];
#pragma unroll
            for (int k = 0; k < CH; ++k) {
                const uint32_t w = w0 + k;
                if (w <= wb) {
                    const int ew = w == wa ? ea : 0;
                    const float4 *sw =
                        reinterpret_cast<const float4 *>(p.slots) + ((size_t)(w * 2 + ew) * 32 + lane) * (2 * NT);
#pragma unroll
                    for (int f = 0; f < 2 * NT; ++f) u[k][f] = __ldcg(sw + f);
                }
            }
#pragma unroll
            for (int k = 0; k < CH; ++k) {
                if (w0 + k <= wb) {
#pragma unroll
                    for (int rt = 0; rt < 2; ++rt)
#pragma unroll
                        for (int j = 0; j < NT; ++j) {
                            const float4 x = u[k][rt * NT + j];
                            v[rt][j][0] += x.x;
                            v[rt][j][1] += x.y;
                            v[rt][j][2] += x.z;
                            v[rt][j][3] += x.w;
                        }
                }
            }
        }
        finish(v, pj, lt, ba0, bu0);
    };

    // ------------------------------------------------ the stream ----------
    zero_acc();
    uint32_t rt = t0 / P, kc = t0 - rt * P;
    Scales cur, nxt;
    load_scales(t0, cur);
    // X^T fragments of one block (k-chunk kc2, block b2), requested one block
    // ahead of their use, so that a read from L2 overlaps a block's decode
    auto load_x = [&](uint32_t kc2, int b2, uint4 (&xv)[NT][2]) {
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            if (xb[j]) {
                const uint4 *xp = reinterpret_cast<const uint4 *>(xb[j] + kc2 * C::TK + b2 * kBlock);
                xv[j][0] = __ldg(xp);
                xv[j][1] = __ldg(xp + 1);
            } else {
                xv[j][0] = xv[j][1] = make_uint4(0, 0, 0, 0);
            }
        }
    };
    constexpr bool kXpf = true;
    uint4 xcur[NT][2];
    if (kXpf) load_x(kc, 0, xcur);
    for (int i = 0; i < n; ++i) {
        const int s = i % S;
        const uint32_t par = (uint32_t)(i / S) & 1u;
        if (i + 1 < n) load_scales(t0 + i + 1, nxt);
        // every lane waits (each observes the landed bytes); a lane that
        // ran out of time stops the whole warp
        const bool ok = tc_wait(&full[s], par, p.wait_ns, (10u << 16) | 2, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
            // out of time: let this warp's loads in flight land, then stop
            if (lane == 0)
                for (int q = i; q < i + S && q < n; ++q) drain_wait(&full[q % S], (uint32_t)(q / S) & 1u);
            __syncwarp();
            return;
        }
        if (i < 4) QLORA_FEW_STAMP(gw, 2 + 2 * i);
        const uint8_t *sl = sp(slot_of(s));
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            uint4 xv[NT][2], xn[NT][2];
            if (kXpf) {
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    xv[j][0] = xcur[j][0];
                    xv[j][1] = xcur[j][1];
                }
                // the next block's fragments: this task's block b + 1, or the
                // next task's first block (k-chunk kc + 1, or 0 in a new tile)
                if (b < 3)
                    load_x(kc, b + 1, xn);
                else if (i + 1 < n)
                    load_x(kc + 1 == P ? 0u : kc + 1, 0, xn);
            } else {
                load_x(kc, b, xv);
            }
            uint2 cw[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) cw[q] = *reinterpret_cast<const uint2 *>(sl + code_off(q, b));
            float blk[2][NT][4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                uint32_t a[2][4];  // [row tile][fragment]
#pragma unroll
                for (int r2 = 0; r2 < 2; ++r2) {
                    const uint32_t w0 = kk < 2 ? cw[2 * r2].x : cw[2 * r2].y;      // row 16 r2 + g
                    const uint32_t w1 = kk < 2 ? cw[2 * r2 + 1].x : cw[2 * r2 + 1].y;  // row 16 r2 + 8 + g
                    if (kk & 1) {
                        a[r2][0] = few_lut<2>(w0, lanebase);
                        a[r2][1] = few_lut<2>(w1, lanebase);
                        a[r2][2] = few_lut<3>(w0, lanebase);
                        a[r2][3] = few_lut<3>(w1, lanebase);
                    } else {
                        a[r2][0] = few_lut<0>(w0, lanebase);
                        a[r2][1] = few_lut<0>(w1, lanebase);
                        a[r2][2] = few_lut<1>(w0, lanebase);
                        a[r2][3] = few_lut<1>(w1, lanebase);
                    }
                }
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const uint32_t b0 = kk < 2 ? (kk == 0 ? xv[j][0].x : xv[j][0].z)
                                               : (kk == 2 ? xv[j][1].x : xv[j][1].z);
                    const uint32_t b1 = kk < 2 ? (kk == 0 ? xv[j][0].y : xv[j][0].w)
                                               : (kk == 2 ? xv[j][1].y : xv[j][1].w);
#pragma unroll
                    for (int r2 = 0; r2 < 2; ++r2) {
                        if (kk == 0)
                            few_mma_z(blk[r2][j], a[r2], b0, b1);
                        else
                            few_mma(blk[r2][j], a[r2], b0, b1);
                    }
                }
            }
            // block scale a' of rows g + 8 q
            float ap[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (F32A) {
                    ap[q] = b == 0 ? cur.a[q].x : (b == 1 ? cur.a[q].y : (b == 2 ? cur.a[q].z : cur.a[q].w));
                } else {
                    ap[q] = dq_absmax((int8_t)((cur.q[q] >> (8 * b)) & 0xFFu), cur.s2[q], MULTI ? cur.mean : mean0);
                }
            }
#pragma unroll
            for (int r2 = 0; r2 < 2; ++r2)
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    acc[r2][j][0] = fmaf(ap[2 * r2], blk[r2][j][0], acc[r2][j][0]);
                    acc[r2][j][1] = fmaf(ap[2 * r2], blk[r2][j][1], acc[r2][j][1]);
                    acc[r2][j][2] = fmaf(ap[2 * r2 + 1], blk[r2][j][2], acc[r2][j][2]);
                    acc[r2][j][3] = fmaf(ap[2 * r2 + 1], blk[r2][j][3], acc[r2][j][3]);
                }
            if (kXpf)
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    xcur[j][0] = xn[j][0];
                    xcur[j][1] = xn[j][1];
                }
        }
        if (i < 4) QLORA_FEW_STAMP(gw, 3 + 2 * i);
        // every lane is done with the slot: refill it
        __syncwarp();
        if (lane == 0 && i + S < n) {
            fence_proxy_async_smem();
            issue(s, t0 + i + S);
        }
        if (kc + 1 == P || i + 1 == n) {
            end_tile(rt);
            if (n_end < 2) QLORA_FEW_STAMP(gw, 11 + 2 * n_end);
            ++n_end;
            zero_acc();
        }
        if (++kc == P) {
            kc = 0;
            ++rt;
        }
        cur = nxt;
    }
    QLORA_FEW_STAMP(gw, 14);
#ifdef QLORA_GEMM_STAMPS
    if (lane == 0) d_few_stamps[gw][15] = (unsigned long long)n_fin;
#endif
}

}  // namespace qlora
