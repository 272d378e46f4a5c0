// fwd_few.cuh -- forward of the NF4 LoRA linear layer for a few tokens
// (M <= 16, decode-like), bound by streaming the packed weight from HBM.
//
//   Y [M, N] = X [M, K] . W'^T + (sU) [M, r] . B^T          (K % 1024 == 0)
//
// Work: the weight is cut into stages of 32 rows x 1024 k (16 blocks of 64)
// in row-group-major order, and every stage into 8 slices of two blocks (one
// per compute warp). The slices form one line that is split evenly over a
// persistent grid: CTA c takes slices [c T / G, (c + 1) T / G), so every CTA
// streams the same number of weights, up to one slice.
//
// Per CTA: one TMA warp streams each stage's code slices (32 rows x 64 bytes,
// 64-byte swizzle; only the slices in the CTA's range) and the stage's int8
// absmax codes (32 rows x 16 bytes) through a ring; eight compute warps each
// take one slice per stage. A warp expands its codes through a byte-indexed
// table in shared memory -- entry b holds the bf16 pair (L[b >> 4], L[b & 15])
// of the two codes a byte packs, one copy of the 256 entries per lane so that
// a warp's 32 lookups hit 32 different banks -- straight into the A fragments
// of mma.sync m16n8k16 (two 16-row tiles), multiplies them with X^T fragments
// (k permuted identically in A and X inside each block), and scales each
// block's fp32 sum by the block's reconstructed absmax
// a' = fp32(q) * scale + mean, so a weight enters as bf16(L[code]) * a'
// (within one bf16 rounding of bf16(L[code] * a')).
//
// When a 32-row group ends, the eight warps' sums meet in shared memory in
// warp order. After the streaming loop (and after the LoRA down-projection
// that precedes this kernel has finished: programmatic dependent launch), each
// row group is finished: held whole by this CTA, its outputs get the LoRA term
// sum_j sU[m, j] B[n, j] and are written as bf16; shared with neighbouring
// CTAs (at most the first and the last group of a CTA), its fp32 partial goes
// to this CTA's slot and an arrival counter is bumped; the CTA that arrives
// last adds all partials in CTA order and writes the outputs. Nothing waits on
// another CTA.
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
    static constexpr int WARPS = 8;                     // compute warps, one slice of two blocks each
    static constexpr int THREADS = 32 * (WARPS + 1);    // + the TMA warp
    static constexpr int SLICE_BYTES = ROWS * 64;       // 32 rows x 64 bytes of codes
    static constexpr int Q_BYTES = ROWS * 16;           // the stage's int8 absmax codes
    static constexpr int STAGE_BYTES = WARPS * SLICE_BYTES + Q_BYTES;
    static constexpr int STAGES = 5;
    static constexpr int MAX_NT = 2;                    // 8-token tiles: up to 16 tokens
    static constexpr int SUM_FLOATS = ROWS * 8 * MAX_NT;  // one row group's sums [32][16]
    static constexpr int MAX_GROUPS = 16;               // row groups one CTA may touch
    static constexpr int B_BYTES = 32768;               // the CTA's rows of the LoRA B (bf16)
    static constexpr int SU_FLOATS = 16 * 128;          // s*U [M <= 16][r <= 128] as fp32
    static constexpr int TABLE_WORDS = 256 * 32;        // 256 entries x 32 lane copies
    static constexpr int OFF_RING = TABLE_WORDS * 4;
    static constexpr int OFF_RED = OFF_RING + STAGES * STAGE_BYTES;
    static constexpr int OFF_SUM = OFF_RED + 2 * WARPS * SUM_FLOATS * 4;
    static constexpr int OFF_B = OFF_SUM + MAX_GROUPS * SUM_FLOATS * 4;
    static constexpr int OFF_SU = OFF_B + B_BYTES;
    static constexpr int OFF_BAR = OFF_SU + SU_FLOATS * 4;
    static constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;
    static constexpr int GRID = 148;                    // CTAs before the row-group cap (one per SM)
};
static_assert(FewCfg::STAGE_BYTES % 512 == 0 && FewCfg::OFF_RING % 1024 == 0, "64-byte swizzle alignment");
static_assert(FewCfg::SMEM_BYTES <= 232448, "shared memory per CTA");

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
    int64_t slices;        // T = row groups x stages per group x 8
    int64_t spg;           // stages per row group (K / 1024)
    uint64_t wait_ns;
};

// first slice of CTA c on a grid of G
__host__ __device__ __forceinline__ int64_t few_begin(int64_t c, int64_t G, int64_t T) { return c * T / G; }

// the CTA whose slice range holds slice x
__host__ __device__ __forceinline__ int64_t few_cta_of(int64_t x, int64_t G, int64_t T) {
    int64_t c = x * G / T;
    while (c + 1 < G && few_begin(c + 1, G, T) <= x) ++c;
    while (c > 0 && few_begin(c, G, T) > x) --c;
    return c;
}

// 16-byte global -> shared copy that does not block the thread
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Row groups CTA c touches (first, count); count 0 for an empty range.
__host__ __device__ __forceinline__ void few_groups(int64_t c, int64_t G, int64_t T, int64_t spg, int64_t &g0,
                                                    int64_t &ng) {
    const int64_t x0 = few_begin(c, G, T), x1 = few_begin(c + 1, G, T);
    if (x1 <= x0) {
        g0 = 0;
        ng = 0;
        return;
    }
    g0 = x0 / (8 * spg);
    ng = (x1 - 1) / (8 * spg) - g0 + 1;
}

// byte j of v as a byte offset into one lane's column of the table (entry
// stride 128 bytes: 32 lane copies of 4 bytes)
template <int J>
__device__ __forceinline__ uint32_t tab_off(uint32_t v) {
    return J == 0 ? (v << 7) & 0x7F80u : (J == 1 ? (v >> 1) & 0x7F80u : (J == 2 ? (v >> 9) & 0x7F80u : (v >> 17) & 0x7F80u));
}
// (the table is written before the CTA barrier and never again)
__device__ __forceinline__ uint32_t lds_u32(uint32_t saddr) {
    uint32_t v;
    asm("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(saddr));
    return v;
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
template <int NT>
__global__ void __launch_bounds__(FewCfg::THREADS, 1)
    k_fwd_few(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_q,
              const FewParams p) {
    using C = FewCfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint32_t *table = reinterpret_cast<uint32_t *>(smem);
    uint8_t *ring = smem + C::OFF_RING;
    float *red = reinterpret_cast<float *>(smem + C::OFF_RED);   // [2][WARPS][32][8 NT]
    float *gsum = reinterpret_cast<float *>(smem + C::OFF_SUM);  // [MAX_GROUPS][32][8 NT]
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *empty = full + C::STAGES;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + C::STAGES);
    volatile int *bcast = reinterpret_cast<volatile int *>(empty + C::STAGES) + 1;  // two words
    constexpr int SF = C::ROWS * 8 * NT;  // floats of one row group's sums

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t G = gridDim.x, c = blockIdx.x, T = p.slices, spg = p.spg;
    const int64_t x0 = few_begin(c, G, T), x1 = few_begin(c + 1, G, T);
    const int64_t st0 = x0 / 8, st1 = x1 > x0 ? (x1 + 7) / 8 : st0;  // stages touched
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

    // the TMA warp: stage st -> ring slot (st - st0) % STAGES
    auto issue = [&](int64_t st) {
        const int s = (int)((st - st0) % C::STAGES);
        const int64_t rg = st / spg, kc = st - rg * spg;
        int nsl = 0;
        for (int w = 0; w < C::WARPS; ++w) {
            const int64_t x = st * 8 + w;
            nsl += (x >= x0 && x < x1) ? 1 : 0;
        }
        uint8_t *base = ring + s * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&full[s], (uint32_t)(nsl * C::SLICE_BYTES + C::Q_BYTES));
        for (int w = 0; w < C::WARPS; ++w) {
            const int64_t x = st * 8 + w;
            if (x >= x0 && x < x1)
                tma_load_2d(base + w * C::SLICE_BYTES, &tm_codes, &full[s], (int32_t)(kc * 512 + 64 * w),
                            (int32_t)(rg * C::ROWS));
        }
        tma_load_2d(base + C::WARPS * C::SLICE_BYTES, &tm_q, &full[s], (int32_t)(kc * 16), (int32_t)(rg * C::ROWS));
    };
    if (warp == C::WARPS && lane == 0) {
        prefetch_tmap(&tm_codes);
        prefetch_tmap(&tm_q);
        for (int64_t st = st0; st < st1 && st < st0 + C::STAGES; ++st) issue(st);
    }
    // the byte table: word (e * 32 + l) = bf16 pair (L[e >> 4] low, L[e & 15] high)
    for (int i = threadIdx.x; i < C::TABLE_WORDS; i += C::THREADS) {
        const int e = i >> 5;
        table[i] = pack_bf16x2(c_levels[e >> 4], c_levels[e & 15]);
    }
    __syncthreads();

    if (warp == C::WARPS) {
        // ------------------------------------------------ TMA producer ----
        if (lane == 0) {
            int64_t issued = st1 - st0 < C::STAGES ? st1 - st0 : C::STAGES;
            for (int64_t st = st0 + C::STAGES; st < st1; ++st) {
                const int s = (int)((st - st0) % C::STAGES);
                const uint32_t u = (uint32_t)((st - st0) / C::STAGES);
                if (!tc_wait(&empty[s], (u - 1) & 1, p.wait_ns, (10u << 16) | 1, abort_flag)) break;
                issue(st);
                issued = st - st0 + 1;
            }
            // every load issued has landed before the CTA moves on
            for (int s = 0; s < C::STAGES && s < issued; ++s) {
                const int64_t last = issued - 1 - ((issued - 1 - s) % C::STAGES);
                drain_wait(&full[s], (uint32_t)(last / C::STAGES) & 1);
            }
        }
    } else {
        // -------------------------------------------- compute warps 0..7 ----
        const int g = lane >> 2, t = lane & 3;
        const uint32_t tab = smem_u32(table) + 4u * lane;
        const float mean = *p.mean;
        // this thread's 8 code bytes of block b of its slice, row g (+ 8 i: +512 i)
        uint32_t coff[2];
#pragma unroll
        for (int b = 0; b < 2; ++b)
            coff[b] = (uint32_t)(g * 64 + ((((2 * b + (t >> 1)) ^ ((g >> 1) & 3))) << 4) + (t & 1) * 8);
        // X^T fragments of block kb: token 8 j + g, k = 64 kb + 16 t .. + 15
        auto load_x = [&](int64_t kb, uint4 (&xv)[NT][2]) {
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int64_t m = 8 * j + g;
                if (m < p.M) {
                    const uint4 *xp = reinterpret_cast<const uint4 *>(p.X + m * p.K + kb * kBlock + 16 * t);
                    xv[j][0] = __ldg(xp);
                    xv[j][1] = __ldg(xp + 1);
                } else {
                    xv[j][0] = xv[j][1] = make_uint4(0, 0, 0, 0);
                }
            }
        };
        // second-level scales of rows g + 8 i for stage st (one per row: a
        // stage's 16 blocks of a row lie in one group of 256)
        auto load_s2 = [&](int64_t st, float (&sv)[4]) {
            const int64_t rg = st / spg, kc = st - rg * spg;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int64_t n = rg * C::ROWS + g + 8 * i;
                sv[i] = n < p.N ? __ldg(p.s2 + ((n * kblocks + kc * 16) >> 8)) : 0.0f;
            }
        };
        float acc[2][NT][4];
        auto zero_acc = [&]() {
#pragma unroll
            for (int rt = 0; rt < 2; ++rt)
#pragma unroll
                for (int j = 0; j < NT; ++j) acc[rt][j][0] = acc[rt][j][1] = acc[rt][j][2] = acc[rt][j][3] = 0.0f;
        };
        // the eight warps' sums of a finished row group, added in warp order
        auto flush = [&](int rl) {
            float *rb = red + (rl & 1) * C::WARPS * SF + warp * SF;
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
            const float *rs = red + (rl & 1) * C::WARPS * SF;
            for (int i = threadIdx.x; i < SF; i += C::WARPS * 32) {
                float v = rs[i];
#pragma unroll
                for (int w = 1; w < C::WARPS; ++w) v += rs[w * SF + i];
                gsum[rl * SF + i] = v;
            }
        };

        // After an abort a warp keeps walking the stages without waiting or
        // working, so that all eight warps reach the same row-group barriers.
        bool alive = true;
        int64_t cur = st0 < st1 ? st0 / spg : 0;
        int rl = 0;
        zero_acc();
        uint4 xv[NT][2], xn[NT][2];
        float sv[4], sn[4];
        {
            const int64_t kc = st0 - (st0 / spg) * spg;
            load_x(kc * 16 + 2 * warp, xv);
            load_s2(st0, sv);
        }
        for (int64_t st = st0; st < st1; ++st) {
            const int64_t rg = st / spg, kc = st - rg * spg;
            if (rg != cur) {
                flush(rl);
                ++rl;
                cur = rg;
                zero_acc();
            }
            const int s = (int)((st - st0) % C::STAGES);
            const int64_t x = st * 8 + warp;
            const bool mine = x >= x0 && x < x1;
            if (alive && !tc_wait(&full[s], (uint32_t)((st - st0) / C::STAGES) & 1, p.wait_ns, (10u << 16) | 2,
                                  abort_flag))
                alive = false;
            if (!alive) continue;
            const uint8_t *sl = ring + s * C::STAGE_BYTES + warp * C::SLICE_BYTES;
            const int8_t *qt = reinterpret_cast<const int8_t *>(ring + s * C::STAGE_BYTES + C::WARPS * C::SLICE_BYTES);
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                // the next block's X fragments (the next stage's after block 1)
                if (b == 0) {
                    load_x(kc * 16 + 2 * warp + 1, xn);
                } else if (st + 1 < st1) {
                    const int64_t kn = (st + 1) - ((st + 1) / spg) * spg;
                    load_x(kn * 16 + 2 * warp, xn);
                    load_s2(st + 1, sn);
                }
                if (mine) {
                    uint2 cw[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) cw[i] = *reinterpret_cast<const uint2 *>(sl + coff[b] + 512 * i);
                    float blk[2][NT][4];
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        uint32_t a[2][4];
#pragma unroll
                        for (int rt = 0; rt < 2; ++rt) {
                            const uint32_t w0 = kk < 2 ? cw[2 * rt].x : cw[2 * rt].y;
                            const uint32_t w1 = kk < 2 ? cw[2 * rt + 1].x : cw[2 * rt + 1].y;
                            if (kk & 1) {
                                a[rt][0] = lds_u32(tab + tab_off<2>(w0));
                                a[rt][1] = lds_u32(tab + tab_off<2>(w1));
                                a[rt][2] = lds_u32(tab + tab_off<3>(w0));
                                a[rt][3] = lds_u32(tab + tab_off<3>(w1));
                            } else {
                                a[rt][0] = lds_u32(tab + tab_off<0>(w0));
                                a[rt][1] = lds_u32(tab + tab_off<0>(w1));
                                a[rt][2] = lds_u32(tab + tab_off<1>(w0));
                                a[rt][3] = lds_u32(tab + tab_off<1>(w1));
                            }
                        }
#pragma unroll
                        for (int j = 0; j < NT; ++j) {
                            const uint32_t xs[8] = {xv[j][0].x, xv[j][0].y, xv[j][0].z, xv[j][0].w,
                                                    xv[j][1].x, xv[j][1].y, xv[j][1].z, xv[j][1].w};
#pragma unroll
                            for (int rt = 0; rt < 2; ++rt) {
                                if (kk == 0)
                                    mma_bf16_16816_z(blk[rt][j], a[rt], xs[0], xs[1]);
                                else
                                    mma_bf16_16816(blk[rt][j], a[rt], xs[2 * kk], xs[2 * kk + 1]);
                            }
                        }
                    }
                    // block scale a' of rows g + 8 i
                    float ap[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) ap[i] = dq_absmax(qt[(g + 8 * i) * 16 + 2 * warp + b], sv[i], mean);
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
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    xv[j][0] = xn[j][0];
                    xv[j][1] = xn[j][1];
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) sv[i] = sn[i];
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        if (st0 < st1) flush(rl);
    }
    __syncthreads();

    // ------------------------------------------------ finishing ----------
    // launched as a programmatic dependent of the kernel that writes sU and
    // zeroes the counters: everything above ran alongside it
    asm volatile("griddepcontrol.wait;" ::: "memory");
    float *sUf = reinterpret_cast<float *>(smem + C::OFF_SU);
    for (int i = threadIdx.x; i < p.M * p.r; i += C::THREADS) {
        const int m = i / p.r, jj = i - m * p.r;
        sUf[i] = bf16lo_to_f32(p.sU[(int64_t)m * p.ldu + jj]);
    }
    // Row groups shared with other CTAs (only the first and the last can
    // be): this CTA's partial goes to its slot (0: its first group, 1: its
    // last), then one arrival per group; the last CTA to arrive finishes it.
    int64_t cf[2] = {0, 0}, cl[2] = {0, 0};
    bool split[2] = {false, false};
    for (int e = 0; e < 2 && e < ng; ++e) {
        const int64_t rg = e == 0 ? g0 : g0 + ng - 1;
        cf[e] = few_cta_of(rg * 8 * spg, G, T);
        cl[e] = few_cta_of((rg + 1) * 8 * spg - 1, G, T);
        split[e] = cl[e] > cf[e];
        if (split[e]) {
            const float *mine = gsum + (e == 0 ? 0 : ng - 1) * SF;
            float *slot = p.slots + (c * 2 + e) * C::SUM_FLOATS;
            for (int i = threadIdx.x; i < SF; i += C::THREADS) __stcg(slot + i, mine[i]);
        }
    }
    __threadfence();
    cp_async_wait_all();
    __syncthreads();
    if (threadIdx.x == 0 && split[0]) bcast[0] = (int)atomicAdd(p.counters + g0, 1u);
    if (threadIdx.x == 32 && split[1]) bcast[1] = (int)atomicAdd(p.counters + g0 + ng - 1, 1u);
    __syncthreads();
    const bool fin0 = !split[0] || bcast[0] == (int)(cl[0] - cf[0]);
    const bool fin1 = !split[1] || bcast[1] == (int)(cl[1] - cf[1]);
    if (split[0] || split[1]) __threadfence();
    // every output this CTA finishes, all groups at once
    const int per = C::ROWS * (int)p.M;
    for (int64_t o = threadIdx.x; o < ng * per; o += C::THREADS) {
        const int rl = (int)(o / per);
        const int rem = (int)(o - (int64_t)rl * per);
        const int m = rem >> 5, row = rem & (C::ROWS - 1);
        const int64_t rg = g0 + rl, n = rg * C::ROWS + row;
        if (n >= p.N) continue;
        const int e = rl == 0 ? 0 : (rl == ng - 1 ? 1 : -1);
        const bool shared = e >= 0 && split[e];
        if (shared && !(e == 0 ? fin0 : fin1)) continue;
        const int idx = row * 8 * NT + m;
        float v;
        if (shared) {
            // partials in CTA order (this CTA's from shared memory)
            v = 0.0f;
            for (int64_t cc = cf[e]; cc <= cl[e]; ++cc) {
                float part;
                if (cc == c) {
                    part = gsum[rl * SF + idx];
                } else {
                    int64_t h0, hn;
                    few_groups(cc, G, T, spg, h0, hn);
                    part = __ldcg(p.slots + (cc * 2 + (rg == h0 ? 0 : 1)) * C::SUM_FLOATS + idx);
                }
                v = cc == cf[e] ? part : v + part;
            }
        } else {
            v = gsum[rl * SF + idx];
        }
        float l = 0.0f;
        const uint16_t *brow = sB + (n - nB0) * p.r;
        const float *urow = sUf + m * p.r;
        for (int jj = 0; jj < p.r; ++jj) l = fmaf(urow[jj], bf16lo_to_f32(brow[jj]), l);
        p.Y[(int64_t)m * p.N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(v + l));
    }
}

}  // namespace qlora
