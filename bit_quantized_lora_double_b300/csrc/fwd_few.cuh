// fwd_few.cuh -- forward of the NF4 LoRA linear layer for a few tokens
// (M <= 16, decode-like), bound by streaming the packed weight from HBM.
//
//   Y [M, N] = X [M, K] . W'^T + (sU) [M, r] . B^T          (K % 1024 == 0)
//
// Work: the weight is cut into stages of 32 rows x 1024 k in row-group-major
// order, and every stage into 16 slices of one block (32 rows x 64 k). The
// slices form one line that is split evenly over a persistent grid: CTA c
// takes slices [c T / G, (c + 1) T / G), so every CTA streams the same number
// of weights, up to one slice.
//
// Per CTA: one TMA warp streams each stage's codes (four boxes of 32 rows x 128
// bytes, 128-byte swizzle; only the boxes holding slices of the CTA's range)
// and its int8 absmax codes (32 rows x 16 bytes) through a ring, issuing a
// whole stage with one warp instruction; sixteen compute warps each take one
// slice per stage. A warp expands its codes through a byte-indexed
// table in shared memory -- entry b holds the bf16 pair (L[b >> 4], L[b & 15])
// of the two codes a byte packs, one copy of the 256 entries per lane so that
// a warp's 32 lookups hit 32 different banks -- straight into the A fragments
// of mma.sync m16n8k16 (two 16-row tiles), multiplies them with X^T fragments
// (k permuted identically in A and X inside each block), and scales each
// block's fp32 sum by the block's reconstructed absmax
// a' = fp32(q) * scale + mean, so a weight enters as bf16(L[code]) * a'
// (within one bf16 rounding of bf16(L[code] * a')).
//
// When a 32-row group ends, the sixteen warps' sums meet in shared memory in
// warp order. After the streaming loop (and after the LoRA down-projection
// that precedes this kernel has finished: programmatic dependent launch), each
// row group is finished: held whole by this CTA, its outputs get the LoRA term
// sum_j sU[m, j] B[n, j] (B's rows arrive in shared memory during the loop)
// and are written as bf16; shared with neighbouring CTAs (at most the first
// and the last group of a CTA), its fp32 partial goes to this CTA's slot and
// an arrival counter is bumped; the CTA that arrives last adds all partials in
// CTA order and writes the outputs. Nothing waits on another CTA.
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
    static constexpr int ROWS = 32;                     // weight rows per stage (two m16 tiles)
    static constexpr int KSTAGE = 1024;                 // k per stage: 16 blocks
    static constexpr int WARPS = 16;                    // compute warps, one slice (block) each
    static constexpr int THREADS = 32 * (WARPS + 1);    // + the TMA warp
    static constexpr int BOX_BYTES = ROWS * 128;        // one TMA box: 32 rows x 128 bytes (4 slices)
    static constexpr int BOXES = 4;                     // boxes per stage
    static constexpr int STAGE_BYTES = BOXES * BOX_BYTES;  // codes of a stage (16 KB)
    static constexpr int Q_BYTES = ROWS * 16;           // the stage's int8 absmax codes
    static constexpr int STAGES = 5;
    static constexpr int MAX_NT = 2;                    // 8-token tiles: up to 16 tokens
    static constexpr int SUM_FLOATS = ROWS * 8 * MAX_NT;  // one row group's sums [32][16]
    static constexpr int MAX_GROUPS = 16;               // row groups one CTA may touch
    static constexpr int B_BYTES = 32768;               // the CTA's rows of the LoRA B (bf16)
    static constexpr int SU_FLOATS = 16 * 128;          // s*U [M <= 16][r <= 128] as fp32
    static constexpr int TABLE_WORDS = 256 * 32;        // 256 entries x 32 lane copies (static)
    static constexpr int OFF_RING = 0;                  // codes, 1024-byte aligned stages (128-byte swizzle)
    static constexpr int OFF_QRING = OFF_RING + STAGES * STAGE_BYTES;
    static constexpr int OFF_RED = OFF_QRING + STAGES * Q_BYTES;
    static constexpr int OFF_SUM = OFF_RED + WARPS * SUM_FLOATS * 4;
    static constexpr int OFF_B = OFF_SUM + MAX_GROUPS * SUM_FLOATS * 4;
    static constexpr int OFF_SU = OFF_B + B_BYTES;
    static constexpr int OFF_BAR = OFF_SU + SU_FLOATS * 4;
    static constexpr int OFF_LAY = OFF_BAR + 256;       // finishing layout: 4 + 2 x 32 + 32 int64
    static constexpr int SMEM_BYTES = OFF_LAY + 800 + 1024;   // dynamic part
    static constexpr int GRID = 148;                    // CTAs before the row-group cap (one per SM)
};
static_assert(FewCfg::STAGE_BYTES % 1024 == 0, "128-byte swizzle alignment of the stages");
static_assert(FewCfg::BOXES * 4 == FewCfg::WARPS, "one 32-byte block column per warp");
static_assert((4 + 64 + FewCfg::WARPS * FewCfg::SUM_FLOATS / (FewCfg::ROWS * 8)) * 8 <= 800, "finishing layout area");
static_assert(FewCfg::SMEM_BYTES + FewCfg::TABLE_WORDS * 4 <= 232448, "shared memory per CTA");

struct FewParams {
    const uint16_t *X;
    int64_t M, N, K;
    const float *s2;
    const float *mean;
    const uint16_t *sU;   // bf16(s * U) [M, ldu]
    int ldu;
    const uint16_t *B;    // [N, r]
    int r;
    uint16_t *Y;
    float *slots;          // [gridDim.x][2][SUM_FLOATS]: partials of the shared row groups
    uint32_t *counters;    // [ceil(N / 32)], zeroed by the preceding kernel
    int64_t slices;        // T = row groups x stages per group x 16
    int64_t spg;           // stages per row group (K / 1024)
    uint64_t wait_ns;
};

// first slice of CTA c on a grid of G (32-bit arithmetic when c * T fits:
// every realistic shape; the divisions sit on the kernel's critical path)
__host__ __device__ __forceinline__ int64_t few_begin(int64_t c, int64_t G, int64_t T) {
    if (T * G < (int64_t(1) << 32)) return (int64_t)((uint32_t)(c * T) / (uint32_t)G);
    return c * T / G;
}

// the CTA whose slice range holds slice x
__host__ __device__ __forceinline__ int64_t few_cta_of(int64_t x, int64_t G, int64_t T) {
    int64_t c = T * G < (int64_t(1) << 32) ? (int64_t)((uint32_t)(x * G) / (uint32_t)T) : x * G / T;
    while (c + 1 < G && few_begin(c + 1, G, T) <= x) ++c;
    while (c > 0 && few_begin(c, G, T) > x) --c;
    return c;
}

// Row groups CTA c touches (first, count); count 0 for an empty range.
__host__ __device__ __forceinline__ void few_groups(int64_t c, int64_t G, int64_t T, int64_t spg, int64_t &g0,
                                                    int64_t &ng) {
    const int64_t x0 = few_begin(c, G, T), x1 = few_begin(c + 1, G, T);
    if (x1 <= x0) {
        g0 = 0;
        ng = 0;
        return;
    }
    const uint32_t per = (uint32_t)(FewCfg::WARPS * spg);  // slices per row group (< 2^31: host check)
    if (x1 < (int64_t(1) << 32)) {
        g0 = (uint32_t)x0 / per;
        ng = (uint32_t)(x1 - 1) / per - g0 + 1;
    } else {
        g0 = x0 / per;
        ng = (x1 - 1) / per - g0 + 1;
    }
}

// 16-byte global -> shared copy that does not block the thread
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// byte j of v as a byte offset into the table (entry stride 128 bytes: 32
// lane copies of 4 bytes), or-ed with this lane's 4-byte column
template <int J>
__device__ __forceinline__ uint32_t tab_off(uint32_t v, uint32_t lane4) {
    const uint32_t sh = J == 0 ? (v << 7) : (J == 1 ? (v >> 1) : (J == 2 ? (v >> 9) : (v >> 17)));
    return (sh & 0x7F80u) | lane4;
}

// D = A * B (no accumulator input)
__device__ __forceinline__ void mma_bf16_16816_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%10, %10, %10, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}

// NT = number of 8-token tiles (M <= 8 * NT <= 16).
// F32A: the block absmax is stored as fp32 (`absmax`, one per block) instead
// of double-quantized; tab selects the level table (kTableNF4 / kTableINT4).
template <int NT, bool F32A>
__global__ void __launch_bounds__(FewCfg::THREADS, 1)
    k_fwd_few(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_q,
              const FewParams p, const float *__restrict__ absmax, int tab) {
    using C = FewCfg;
    // the byte table: word (e * 32 + l) = bf16 pair (L[e >> 4] low, L[e & 15]
    // high); static, so its base is an immediate of every lookup
    __shared__ uint32_t s_table[C::TABLE_WORDS];
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *ring = smem + C::OFF_RING;
    float *red = reinterpret_cast<float *>(smem + C::OFF_RED);   // [WARPS][32][8 NT]
    float *gsum = reinterpret_cast<float *>(smem + C::OFF_SUM);  // [MAX_GROUPS][32][8 NT]
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *empty = full + C::STAGES;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + C::STAGES);
    volatile int *bcast = reinterpret_cast<volatile int *>(empty + C::STAGES) + 1;  // two words
    volatile int64_t *lay = reinterpret_cast<volatile int64_t *>(smem + C::OFF_LAY);  // finishing layout
    constexpr int SF = C::ROWS * 8 * NT;  // floats of one row group's sums

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t G = gridDim.x, c = blockIdx.x, T = p.slices, spg = p.spg;
    const int64_t x0 = few_begin(c, G, T), x1 = few_begin(c + 1, G, T);
    const int64_t st0 = x0 / C::WARPS;                                   // first stage touched
    const int nst = x1 > x0 ? (int)((x1 + C::WARPS - 1) / C::WARPS - st0) : 0;  // stages touched
    const int wfirst = (int)(x0 - st0 * C::WARPS);                       // first slice in stage 0
    const int wlast = nst > 0 ? (int)(x1 - (st0 + nst - 1) * C::WARPS) : 0;  // slices in the last stage
    const int64_t kblocks = p.K / kBlock;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], C::WARPS);
        }
        *abort_flag = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    // this CTA's rows of B (rows of its row groups, contiguous in B) start
    // coming in now; they are needed only when the outputs are finished
    int64_t g0, ng;
    few_groups(c, G, T, spg, g0, ng);
    const int64_t nB0 = g0 * C::ROWS, nB1 = p.N < (g0 + ng) * C::ROWS ? p.N : (g0 + ng) * C::ROWS;
    uint16_t *sB = reinterpret_cast<uint16_t *>(smem + C::OFF_B);
    {
        const int64_t nbytes = nB1 > nB0 ? (nB1 - nB0) * p.r * 2 : 0;  // <= B_BYTES (host plan)
        const uint8_t *src = reinterpret_cast<const uint8_t *>(p.B + nB0 * p.r);  // 16-byte aligned: nB0 % 32 == 0
        for (int64_t i = threadIdx.x; i < nbytes / 16; i += C::THREADS)
            cp_async16(reinterpret_cast<uint8_t *>(sB) + 16 * i, src + 16 * i);
        for (int64_t i = (nbytes / 16) * 8 + threadIdx.x; i < nbytes / 2; i += C::THREADS)
            sB[i] = p.B[nB0 * p.r + i];
    }
    __syncthreads();

    // The TMA warp issues a stage with one instruction: lane 0 expects the
    // bytes, lanes 0..3 load the 128-byte code boxes that hold slices of this
    // CTA's range, lane 4 the absmax codes.
    uint8_t *qring = smem + C::OFF_QRING;
    auto issue = [&](int i, int s, int64_t rg, int64_t kc) {
        const int wa = i == 0 ? wfirst : 0, wb = i == nst - 1 ? wlast : C::WARPS;
        const int ba = wa >> 2, bb = (wb + 3) >> 2;
        const uint32_t qbytes = F32A ? 0u : (uint32_t)C::Q_BYTES;
        if (lane == 0) mbar_arrive_expect_tx(&full[s], (uint32_t)((bb - ba) * C::BOX_BYTES) + qbytes);
        __syncwarp();
        if (lane >= ba && lane < bb)
            tma_load_2d(ring + s * C::STAGE_BYTES + lane * C::BOX_BYTES, &tm_codes, &full[s],
                        (int32_t)(kc * 512 + 128 * lane), (int32_t)(rg * C::ROWS));
        if (lane == 4 && !F32A)
            tma_load_2d(qring + s * C::Q_BYTES, &tm_q, &full[s], (int32_t)(kc * 16), (int32_t)(rg * C::ROWS));
    };
    int64_t prg = (uint32_t)st0 / (uint32_t)spg, pkc = st0 - prg * spg;  // the producer's next stage
    auto pnext = [&]() {
        if (++pkc == spg) {
            pkc = 0;
            ++prg;
        }
    };
    if (warp == C::WARPS) {
        if (lane == 0) {
            prefetch_tmap(&tm_codes);
            prefetch_tmap(&tm_q);
        }
        for (int i = 0; i < nst && i < C::STAGES; ++i) {
            issue(i, i, prg, pkc);
            pnext();
        }
    }
    for (int i = threadIdx.x; i < C::TABLE_WORDS; i += C::THREADS) {
        const int e = i >> 5;
        s_table[i] = pack_bf16x2(c_levels_q4[tab][e >> 4], c_levels_q4[tab][e & 15]);
    }
    __syncthreads();

    if (warp == C::WARPS) {
        // ------------------------------------------------ TMA producer ----
        int issued = nst < C::STAGES ? nst : C::STAGES;
        int s = 0;
        uint32_t ph = 0;
        for (int i = C::STAGES; i < nst; ++i) {
            int ok = 1;
            if (lane == 0) ok = tc_wait(&empty[s], ph, p.wait_ns, (10u << 16) | 1, abort_flag) ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, ok, 0)) break;
            issue(i, s, prg, pkc);
            pnext();
            issued = i + 1;
            if (++s == C::STAGES) {
                s = 0;
                ph ^= 1u;
            }
        }
        // every load issued has landed before the CTA moves on
        if (lane == 0)
            for (int q = 0; q < C::STAGES && q < issued; ++q) {
                const int last = issued - 1 - ((issued - 1 - q) % C::STAGES);
                drain_wait(&full[q], (uint32_t)(last / C::STAGES) & 1);
            }
    } else {
        // ------------------------------------------- compute warps 0..15 ----
        // The finishing needs to know which CTAs share this CTA's first and
        // last row groups and which slot each of them writes. Integer
        // divisions with long dependency chains: the lanes of the last
        // compute warp work them out side by side while the first stage is
        // still in flight. Layout: [0..3] first and last CTA sharing the
        // first and the last group; [4 + 32 e + k] the slot of CTA
        // cf[e] + k (-1: this CTA), for up to 32 CTAs per group (more are
        // looked up at the end).
        if (warp == C::WARPS - 1) {
            if (lane < 4) {
                const int e = lane >> 1;
                int64_t v = (lane & 1) ? -1 : 0;  // no such group: cf = 0, cl = -1
                if (e < ng) {
                    const int64_t rg = e == 0 ? g0 : g0 + ng - 1;
                    v = (lane & 1) ? few_cta_of((rg + 1) * C::WARPS * spg - 1, G, T)
                                   : few_cta_of(rg * C::WARPS * spg, G, T);
                }
                lay[lane] = v;
            }
            __syncwarp();
            for (int e = 0; e < 2 && e < ng; ++e) {
                const int64_t a = lay[2 * e], b = lay[2 * e + 1];
                const int64_t rg = e == 0 ? g0 : g0 + ng - 1;
                const int64_t cc = a + lane;
                if (cc <= b) {
                    int64_t h0, hn;
                    few_groups(cc, G, T, spg, h0, hn);
                    lay[4 + 32 * e + lane] = cc == c ? -1 : cc * 2 + (rg == h0 ? 0 : 1);
                }
            }
        }
        const int g = lane >> 2, t = lane & 3;
        const uint32_t lane4 = 4u * lane;
        const char *tab = reinterpret_cast<const char *>(s_table);
        const float mean = F32A ? 0.0f : *p.mean;
        // this thread's 8 code bytes of rows g + 8 q of its block: block
        // column warp & 3 of box warp >> 2 (128-byte rows, 128-byte swizzle:
        // 16-byte chunk h of row r sits at h ^ (r & 7))
        const uint32_t coff = (uint32_t)((warp >> 2) * C::BOX_BYTES + g * 128 +
                                         (((2 * (warp & 3) + (t >> 1)) ^ g) << 4) + (t & 1) * 8);
        // X^T fragments: token 8 j + g, k = 64 kb + 16 t .. + 15
        const uint16_t *xb[NT];
#pragma unroll
        for (int j = 0; j < NT; ++j) xb[j] = 8 * j + g < p.M ? p.X + (8 * j + g) * p.K + 16 * t : nullptr;
        auto load_x = [&](int64_t kb, uint4 (&xv)[NT][2]) {
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                if (xb[j]) {
                    const uint4 *xp = reinterpret_cast<const uint4 *>(xb[j] + kb * kBlock);
                    xv[j][0] = __ldg(xp);
                    xv[j][1] = __ldg(xp + 1);
                } else {
                    xv[j][0] = xv[j][1] = make_uint4(0, 0, 0, 0);
                }
            }
        };
        // second-level scales of rows g + 8 i of a stage (one per row: a
        // stage's 16 blocks of a row lie in one group of 256); sbase[i] is
        // the row's first block index, refreshed per row group (the host
        // keeps N * K / 64 below 2^31 on this path). Rows past the last one
        // read row 0's scale: their sums are never written.
        uint32_t sbase[4];
        auto set_rows = [&](int64_t rg) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int64_t n = rg * C::ROWS + g + 8 * i;
                sbase[i] = n < p.N ? (uint32_t)(n * kblocks) : 0u;
            }
        };
        // (with fp32 absmax: the absmax of this warp's block of rows g + 8 i)
        auto load_s2 = [&](int64_t kc, float (&sv)[4]) {
            const uint32_t k16 = (uint32_t)kc * 16u;
            if (F32A) {
#pragma unroll
                for (int i = 0; i < 4; ++i) sv[i] = __ldg(absmax + sbase[i] + k16 + (uint32_t)warp);
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) sv[i] = __ldg(p.s2 + ((sbase[i] + k16) >> 8));
            }
        };
        float acc[2][NT][4];
        auto zero_acc = [&]() {
#pragma unroll
            for (int rt = 0; rt < 2; ++rt)
#pragma unroll
                for (int j = 0; j < NT; ++j) acc[rt][j][0] = acc[rt][j][1] = acc[rt][j][2] = acc[rt][j][3] = 0.0f;
        };
        // the sixteen warps' sums of a finished row group, added in warp order
        auto flush = [&](int rl) {
            float *rb = red + warp * SF;
#pragma unroll
            for (int rt = 0; rt < 2; ++rt)
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    rb[(16 * rt + g) * 8 * NT + 8 * j + 2 * t] = acc[rt][j][0];
                    rb[(16 * rt + g) * 8 * NT + 8 * j + 2 * t + 1] = acc[rt][j][1];
                    rb[(16 * rt + g + 8) * 8 * NT + 8 * j + 2 * t] = acc[rt][j][2];
                    rb[(16 * rt + g + 8) * 8 * NT + 8 * j + 2 * t + 1] = acc[rt][j][3];
                }
            asm volatile("bar.sync 1, %0;" ::"n"(C::WARPS * 32) : "memory");
            for (int i = threadIdx.x; i < SF; i += C::WARPS * 32) {
                float v = red[i];
#pragma unroll
                for (int w = 1; w < C::WARPS; ++w) v += red[w * SF + i];
                gsum[rl * SF + i] = v;
            }
            asm volatile("bar.sync 1, %0;" ::"n"(C::WARPS * 32) : "memory");
        };

        // After an abort a warp keeps walking the stages without waiting or
        // working, so that all sixteen warps reach the same row-group barriers.
        bool alive = true;
        int64_t rg = (uint32_t)st0 / (uint32_t)spg, kc = st0 - rg * spg;  // stage st0 + i: row group, k-chunk
        int rl = 0, s = 0;
        uint32_t ph = 0;
        zero_acc();
        set_rows(rg);
        auto mine_at = [&](int i) { return !(i == 0 && warp < wfirst) && !(i == nst - 1 && warp >= wlast); };
        // the block scales of a stage are requested one stage ahead (a
        // dependent L2 read in every stage otherwise: ~1 us per stage); the
        // X fragments, L1 hits after the first stages, with the stage itself
        float sv_next[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (nst > 0 && mine_at(0)) load_s2(kc, sv_next);
        for (int i = 0; i < nst; ++i) {
            const bool mine = mine_at(i);
            uint4 xv[NT][2];
            float sv[4] = {sv_next[0], sv_next[1], sv_next[2], sv_next[3]};
            if (alive && mine) load_x(kc * 16 + warp, xv);
            if (alive && !tc_wait(&full[s], ph, p.wait_ns, (10u << 16) | 2, abort_flag)) alive = false;
            if (alive) {
                if (mine) {
                    const uint8_t *sl = ring + s * C::STAGE_BYTES;
                    const int8_t *qt = reinterpret_cast<const int8_t *>(qring + s * C::Q_BYTES);
                    uint2 cw[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) cw[q] = *reinterpret_cast<const uint2 *>(sl + coff + 1024 * q);
                    float blk[2][NT][4];
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        uint32_t a[2][4];  // [row tile][fragment]
#pragma unroll
                        for (int rt = 0; rt < 2; ++rt) {
                            const uint32_t w0 = kk < 2 ? cw[2 * rt].x : cw[2 * rt].y;
                            const uint32_t w1 = kk < 2 ? cw[2 * rt + 1].x : cw[2 * rt + 1].y;
                            if (kk & 1) {
                                a[rt][0] = *reinterpret_cast<const uint32_t *>(tab + tab_off<2>(w0, lane4));
                                a[rt][1] = *reinterpret_cast<const uint32_t *>(tab + tab_off<2>(w1, lane4));
                                a[rt][2] = *reinterpret_cast<const uint32_t *>(tab + tab_off<3>(w0, lane4));
                                a[rt][3] = *reinterpret_cast<const uint32_t *>(tab + tab_off<3>(w1, lane4));
                            } else {
                                a[rt][0] = *reinterpret_cast<const uint32_t *>(tab + tab_off<0>(w0, lane4));
                                a[rt][1] = *reinterpret_cast<const uint32_t *>(tab + tab_off<0>(w1, lane4));
                                a[rt][2] = *reinterpret_cast<const uint32_t *>(tab + tab_off<1>(w0, lane4));
                                a[rt][3] = *reinterpret_cast<const uint32_t *>(tab + tab_off<1>(w1, lane4));
                            }
                        }
#pragma unroll
                        for (int j = 0; j < NT; ++j) {
                            const uint32_t b0 = kk < 2 ? (kk == 0 ? xv[j][0].x : xv[j][0].z)
                                                       : (kk == 2 ? xv[j][1].x : xv[j][1].z);
                            const uint32_t b1 = kk < 2 ? (kk == 0 ? xv[j][0].y : xv[j][0].w)
                                                       : (kk == 2 ? xv[j][1].y : xv[j][1].w);
#pragma unroll
                            for (int rt = 0; rt < 2; ++rt) {
                                if (kk == 0)
                                    mma_bf16_16816_z(blk[rt][j], a[rt], b0, b1);
                                else
                                    mma_bf16_16816(blk[rt][j], a[rt], b0, b1);
                            }
                        }
                    }
                    // block scale a' of rows g + 8 q
                    float ap[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) ap[q] = F32A ? sv[q] : dq_absmax(qt[(g + 8 * q) * 16 + warp], sv[q], mean);
#pragma unroll
                    for (int rt = 0; rt < 2; ++rt)
#pragma unroll
                        for (int j = 0; j < NT; ++j) {
                            acc[rt][j][0] = fmaf(ap[2 * rt], blk[rt][j][0], acc[rt][j][0]);
                            acc[rt][j][1] = fmaf(ap[2 * rt], blk[rt][j][1], acc[rt][j][1]);
                            acc[rt][j][2] = fmaf(ap[2 * rt + 1], blk[rt][j][2], acc[rt][j][2]);
                            acc[rt][j][3] = fmaf(ap[2 * rt + 1], blk[rt][j][3], acc[rt][j][3]);
                        }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
            if (++s == C::STAGES) {
                s = 0;
                ph ^= 1u;
            }
            int64_t rg_n = rg, kc_n = kc + 1;
            if (kc_n == spg) {
                kc_n = 0;
                ++rg_n;
            }
            // a row group ends here when the next stage starts another one
            if (i + 1 == nst || rg_n != rg) {
                flush(rl);
                ++rl;
                zero_acc();
            }
            if (rg_n != rg) set_rows(rg_n);
            if (alive && i + 1 < nst && mine_at(i + 1)) load_s2(kc_n, sv_next);
            rg = rg_n;
            kc = kc_n;
        }
    }
    __syncthreads();

    // ------------------------------------------------ finishing ----------
    // launched as a programmatic dependent of the kernel that writes sU and
    // zeroes the counters (it writes nothing else this kernel reads):
    // everything above ran alongside it
    asm volatile("griddepcontrol.wait;" ::: "memory");
    float *sUf = reinterpret_cast<float *>(smem + C::OFF_SU);
    for (int i = threadIdx.x; i < p.M * p.r; i += C::THREADS) {
        const int m = i / p.r, jj = i - m * p.r;
        sUf[i] = bf16lo_to_f32(p.sU[(int64_t)m * p.ldu + jj]);
    }
    // Row groups shared with other CTAs (only the first and the last can
    // be): this CTA's partial goes to its slot (0: its first group, 1: its
    // last), then one arrival per group; the last CTA to arrive finishes it.
    // (the CTAs sharing them were worked out at the start: `lay`)
    const int64_t cf[2] = {lay[0], lay[2]}, cl[2] = {lay[1], lay[3]};
    const bool split[2] = {ng > 0 && cl[0] > cf[0], ng > 1 && cl[1] > cf[1]};
    for (int e = 0; e < 2; ++e) {
        if (!split[e]) continue;
        const float *mine = gsum + (e == 0 ? 0 : ng - 1) * SF;
        float *slot = p.slots + (c * 2 + e) * C::SUM_FLOATS;
        for (int i = threadIdx.x; i < SF; i += C::THREADS) __stcg(slot + i, mine[i]);
    }
    __threadfence();
    cp_async_wait_all();
    __syncthreads();
    if (threadIdx.x == 0 && split[0]) bcast[0] = (int)atomicAdd(p.counters + g0, 1u);
    if (threadIdx.x == 32 && split[1]) bcast[1] = (int)atomicAdd(p.counters + g0 + ng - 1, 1u);
    __syncthreads();
    const bool fin[2] = {!split[0] || bcast[0] == (int)(cl[0] - cf[0]), !split[1] || bcast[1] == (int)(cl[1] - cf[1])};
    if (split[0] || split[1]) __threadfence();
    // A shared group this CTA finishes: the partials of all its CTAs, added in
    // CTA order, replace this CTA's own in gsum. The other CTAs' slots come in
    // through `red` a chunk of CTAs at a time, every load of a chunk in flight
    // together; the running sum lives in the last SF floats of `red`.
    {
        const int chunk = C::WARPS * C::SUM_FLOATS / SF - 1;
        float *run = red + chunk * SF;
        for (int e = 0; e < 2 && e < ng; ++e) {
            if (!split[e] || !fin[e]) continue;
            const int rl = e == 0 ? 0 : (int)ng - 1;
            const int64_t rg = g0 + rl;
            float *mine = gsum + rl * SF;
            for (int64_t c0 = cf[e]; c0 <= cl[e]; c0 += chunk) {
                const int nc = (int)(cl[e] - c0 + 1 < chunk ? cl[e] - c0 + 1 : chunk);
                // the slot of each CTA of the chunk (-1: this CTA): from the
                // layout for the first 32 CTAs of the group, else looked up
                volatile int64_t *src = lay + 4 + 32 * e + (c0 - cf[e]);
                if (c0 - cf[e] + nc > 32) {
                    src = lay + 4 + 64;
                    if (threadIdx.x < nc) {
                        const int64_t cc = c0 + threadIdx.x;
                        int64_t h0, hn;
                        few_groups(cc, G, T, spg, h0, hn);
                        src[threadIdx.x] = cc == c ? -1 : cc * 2 + (rg == h0 ? 0 : 1);
                    }
                }
                __syncthreads();
                for (int u = threadIdx.x; u < nc * SF; u += C::THREADS) {
                    const int k = u / SF, i = u - k * SF;
                    const int64_t sl = src[k];
                    red[k * SF + i] = sl < 0 ? mine[i] : __ldcg(p.slots + sl * C::SUM_FLOATS + i);
                }
                __syncthreads();
                for (int i = threadIdx.x; i < SF; i += C::THREADS) {
                    float v = c0 == cf[e] ? red[i] : run[i] + red[i];
                    for (int k = 1; k < nc; ++k) v += red[k * SF + i];
                    run[i] = v;
                }
                __syncthreads();
            }
            for (int i = threadIdx.x; i < SF; i += C::THREADS) mine[i] = run[i];
            __syncthreads();
        }
    }
    // every output this CTA finishes, all groups at once: the group's sum
    // plus the LoRA term from shared memory
    const int per = C::ROWS * (int)p.M;
    for (int64_t o = threadIdx.x; o < ng * per; o += C::THREADS) {
        const int rl = (int)(o / per);
        const int rem = (int)(o - (int64_t)rl * per);
        const int m = rem >> 5, row = rem & (C::ROWS - 1);
        const int64_t rg = g0 + rl, n = rg * C::ROWS + row;
        if (n >= p.N) continue;
        const int e = rl == 0 ? 0 : (rl == ng - 1 ? 1 : -1);
        if (e >= 0 && split[e] && !fin[e]) continue;
        const float v = gsum[rl * SF + row * 8 * NT + m];
        float l = 0.0f;
        const uint16_t *brow = sB + (n - nB0) * p.r;
        const float *urow = sUf + m * p.r;
        for (int jj = 0; jj < p.r; ++jj) l = fmaf(urow[jj], bf16lo_to_f32(brow[jj]), l);
        p.Y[(int64_t)m * p.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(v + l));
    }
}

}  // namespace qlora
