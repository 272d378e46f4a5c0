// small_m.cuh -- forward of the NF4 LoRA linear layer for few tokens
// (M <= 32, decode-like), bound by reading the packed weight from HBM.
//
//   Y [M, N] = X [M, K] . W'^T + (sU) [M, r] . B^T
//
// Each CTA (4 compute warps and a TMA warp) owns 16 rows of W, streamed
// through a shared-memory ring in stages of 8 blocks of 64 codes; compute
// warp w takes blocks w and w + 4 of every stage. Per block a thread loads 8 bytes of codes
// for each of two rows (g and g + 8, g = lane / 4), expands them through the
// constant bf16 NF4 table (PRMT byte-plane lookups) straight into the A
// fragments of mma.sync m16n8k16 (W' rows x k) and multiplies with X^T
// fragments (k x tokens) loaded from global memory, 8 tokens per n-tile.
// The 64 k of a block are permuted identically in A and B (thread t of a
// quad holds k = 16 t + 4 c .. + 3 in chunk c), which leaves each block's
// sum unchanged. Each block's fp32 sum is scaled by the block's
// reconstructed absmax a' = fp32(q) * scale + mean, so a weight enters as
// bf16(L[code]) * a' instead of bf16(L[code] * a'): the two differ by at most
// one bf16 rounding of the weight. The four warps' partial sums meet in
// shared memory, in warp order, where the LoRA term is added and Y is
// written as bf16. The kernel is launched as a programmatic dependent of the
// LoRA down-projection and waits for it only before that last step.
// Sources: ashishsrivastav.com "QLoRA: Fine-Tuning a 70B on One GPU", section
// "Double Quantization" (dequantize on the fly); xingyuzhitong.com
// "Fine-Tuning Memory Requirements", section "QLoRA: quantize the frozen base
// to 4 bits".
#pragma once

#include "common.cuh"
#include "gemm_tc.cuh"

namespace qlora {

constexpr int kSmallMaxM = 32;

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

struct SmallCfg {
    static constexpr int ROWS = 16;            // W rows per CTA
    static constexpr int STAGE_BLOCKS = 8;     // 64-wide blocks per stage (two per compute warp)
    static constexpr int STAGE_BYTES = ROWS * STAGE_BLOCKS * 32;  // 4 KB of codes (two 128-byte boxes)
    static constexpr int STAGES = 8;           // 32 KB ring: all of K = 4096 in flight
    static constexpr int THREADS = 160;        // 4 compute warps + 1 TMA warp
};

// Largest K handled by one CTA's table of reconstructed absmax values (the
// caller checks this; 16 rows x 224 blocks x 4 bytes = 14 KB of shared memory).
constexpr int64_t kSmallMaxK = 14336;

// NT = number of 8-token tiles (M <= 8 * NT).
template <int NT>
__global__ void __launch_bounds__(SmallCfg::THREADS) k_fwd_small(const __grid_constant__ CUtensorMap tm_codes,
                                                                 const uint16_t *__restrict__ X, int64_t M, int64_t K,
                                                                 const int8_t *__restrict__ q,
                                                                 const float *__restrict__ s2,
                                                                 const float *__restrict__ mean_p, int64_t N,
                                                                 const uint16_t *__restrict__ sU, int ldu,
                                                                 const uint16_t *__restrict__ B, int r,
                                                                 uint16_t *__restrict__ Y, uint64_t wait_ns,
                                                                 const float *__restrict__ absmax_f32, int tabid) {
    using C = SmallCfg;
    // X^T fragments are prefetched P stages ahead in registers
    constexpr int P = NT == 1 ? 2 : 1;
    __shared__ __align__(1024) uint8_t ring[C::STAGES][C::STAGE_BYTES];
    __shared__ float amax[16][kSmallMaxK / kBlock];
    // the warps' partial sums reuse the ring once every stage is consumed
    float(*red)[16][8 * NT + 1] = reinterpret_cast<float(*)[16][8 * NT + 1]>(&ring[0][0]);
    static_assert(sizeof(float) * 4 * 16 * (8 * NT + 1) <= sizeof(uint8_t) * C::STAGES * C::STAGE_BYTES, "");
    __shared__ uint64_t full[C::STAGES], empty[C::STAGES];
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t n0 = (int64_t)blockIdx.x * C::ROWS;
    const int64_t kblocks = K / kBlock;
    const int64_t nstages = (kblocks + C::STAGE_BLOCKS - 1) / C::STAGE_BLOCKS;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 4);
        }
        abort_flag = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    __syncthreads();
    // the first STAGES code loads go out before anything else
    if (warp == 4 && lane == 0) {
        prefetch_tmap(&tm_codes);
        for (int64_t st = 0; st < nstages && st < C::STAGES; ++st) {
            mbar_arrive_expect_tx(&full[st], C::STAGE_BYTES);
            tma_load_2d(ring[st], &tm_codes, &full[st], (int32_t)(st * C::STAGE_BLOCKS * 32), (int32_t)n0);
            tma_load_2d(ring[st] + 2048, &tm_codes, &full[st], (int32_t)(st * C::STAGE_BLOCKS * 32 + 128),
                        (int32_t)n0);
        }
    }
    // reconstructed absmax a' of every (row, block) of this CTA's 16 rows,
    // while the codes stream in (loads of four entries in flight per thread)
    {
        const float mean = absmax_f32 ? 0.0f : *mean_p;
        const int nb = (int)kblocks, total = 16 * nb;
#pragma unroll 4
        for (int i = threadIdx.x; i < total; i += C::THREADS) {
            const int rr = i / nb, kb = i - rr * nb;
            const int64_t b = (n0 + rr) * kblocks + kb;
            amax[rr][kb] = n0 + rr < N ? (absmax_f32 ? __ldg(absmax_f32 + b) : dq_absmax(__ldg(q + b), __ldg(s2 + (b >> 8)), mean))
                                       : 0.0f;
        }
    }
    __syncthreads();

    float acc[NT][4];
    if (warp == 4) {
        // ------------------------------------------------ TMA producer ----
        if (lane == 0) {
            int64_t issued = nstages < C::STAGES ? nstages : C::STAGES;
            for (int64_t st = C::STAGES; st < nstages; ++st) {
                const int s = (int)(st % C::STAGES);
                const uint32_t u = (uint32_t)(st / C::STAGES);
                if (!tc_wait(&empty[s], (u - 1) & 1, wait_ns, (9u << 16) | 1, &abort_flag)) break;
                mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
                tma_load_2d(ring[s], &tm_codes, &full[s], (int32_t)(st * C::STAGE_BLOCKS * 32), (int32_t)n0);
                tma_load_2d(ring[s] + 2048, &tm_codes, &full[s], (int32_t)(st * C::STAGE_BLOCKS * 32 + 128),
                            (int32_t)n0);
                issued = st + 1;
            }
            // every load issued has landed before the ring is reused for the
            // partial sums (after an abort some were never consumed)
            for (int s = 0; s < C::STAGES && s < issued; ++s) {
                const int64_t last = issued - 1 - ((issued - 1 - s) % C::STAGES);
                drain_wait(&full[s], (uint32_t)(last / C::STAGES) & 1);
            }
        }
    } else {
        // -------------------------------------------- compute warps 0..3 ----
        const int g = lane >> 2, t = lane & 3;
        const Nf4Table tab = make_table(1.0f, tabid);  // bf16(L[i])
        // this thread's 8 code bytes of block `warp` of a stage's box, rows g
        // and g + 8 (128-byte rows, 128-byte swizzle: chunk c at c ^ (row % 8));
        // block warp + 4 sits in the second box, 2048 bytes on
        const uint32_t offA = (uint32_t)(g * 128 + (((2 * warp + (t >> 1)) ^ g) << 4) + (t & 1) * 8);
        const uint32_t offB = offA + 8 * 128;
        // X^T fragments of half h of stage st: token 8 j + g,
        // k = 64 (8 st + 4 h + warp) + 16 t .. + 15
        auto load_x = [&](int64_t st, int h, uint4 (&xv)[NT][2]) {
            const int64_t kb = st * C::STAGE_BLOCKS + 4 * h + warp;
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int64_t m = 8 * j + g;
                if (m < M && kb < kblocks) {
                    const uint4 *xp = reinterpret_cast<const uint4 *>(X + m * K + kb * kBlock + 16 * t);
                    xv[j][0] = __ldg(xp);
                    xv[j][1] = __ldg(xp + 1);
                } else {
                    xv[j][0] = xv[j][1] = make_uint4(0, 0, 0, 0);
                }
            }
        };
        uint4 xbuf[P][2][NT][2];
#pragma unroll
        for (int i = 0; i < P; ++i) {
            load_x(i, 0, xbuf[i][0]);
            load_x(i, 1, xbuf[i][1]);
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
        bool alive = true;
        for (int64_t st0 = 0; st0 < nstages && alive; st0 += P) {
#pragma unroll
            for (int i = 0; i < P; ++i) {
                const int64_t st = st0 + i;
                if (st >= nstages) break;
                const int s = (int)(st % C::STAGES);
                if (!tc_wait(&full[s], (uint32_t)(st / C::STAGES) & 1, wait_ns, (9u << 16) | 2, &abort_flag)) {
                    alive = false;
                    break;
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int64_t kb = st * C::STAGE_BLOCKS + 4 * h + warp;
                    if (kb < kblocks) {
                        const uint2 wa = *reinterpret_cast<const uint2 *>(ring[s] + h * 2048 + offA);
                        const uint2 wb = *reinterpret_cast<const uint2 *>(ring[s] + h * 2048 + offB);
                        const float aA = amax[g][kb], aB = amax[g + 8][kb];
                        uint32_t dA[2][4], dB[2][4];
                        decode8(tab, wa.x, dA[0]);
                        decode8(tab, wa.y, dA[1]);
                        decode8(tab, wb.x, dB[0]);
                        decode8(tab, wb.y, dB[1]);
                        float blk[NT][4];
#pragma unroll
                        for (int j = 0; j < NT; ++j) blk[j][0] = blk[j][1] = blk[j][2] = blk[j][3] = 0.0f;
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            // chunk c: this thread's k = 16 t + 4 c .. + 3 (rows g, g + 8)
                            const uint32_t a[4] = {dA[c >> 1][2 * (c & 1)], dB[c >> 1][2 * (c & 1)],
                                                   dA[c >> 1][2 * (c & 1) + 1], dB[c >> 1][2 * (c & 1) + 1]};
#pragma unroll
                            for (int j = 0; j < NT; ++j) {
                                const uint32_t xs[8] = {xbuf[i][h][j][0].x, xbuf[i][h][j][0].y, xbuf[i][h][j][0].z,
                                                        xbuf[i][h][j][0].w, xbuf[i][h][j][1].x, xbuf[i][h][j][1].y,
                                                        xbuf[i][h][j][1].z, xbuf[i][h][j][1].w};
                                mma_bf16_16816(blk[j], a, xs[2 * c], xs[2 * c + 1]);
                            }
                        }
#pragma unroll
                        for (int j = 0; j < NT; ++j) {
                            acc[j][0] = fmaf(aA, blk[j][0], acc[j][0]);
                            acc[j][1] = fmaf(aA, blk[j][1], acc[j][1]);
                            acc[j][2] = fmaf(aB, blk[j][2], acc[j][2]);
                            acc[j][3] = fmaf(aB, blk[j][3], acc[j][3]);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
                load_x(st + P, 0, xbuf[i][0]);
                load_x(st + P, 1, xbuf[i][1]);
            }
        }
    }
    // the producer's loads have all landed: the ring is free for the partials
    __syncthreads();
    if (warp < 4) {
        // partial sums of this warp: rows g, g + 8; tokens 8 j + 2 t, + 1
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            red[warp][g][8 * j + 2 * t] = acc[j][0];
            red[warp][g][8 * j + 2 * t + 1] = acc[j][1];
            red[warp][g + 8][8 * j + 2 * t] = acc[j][2];
            red[warp][g + 8][8 * j + 2 * t + 1] = acc[j][3];
        }
    }
    __syncthreads();
    // launched as a programmatic dependent of the kernel that writes sU:
    // everything above ran alongside it, its output is visible from here on
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the 16 x M outputs: warp sums in warp order, then the LoRA term
    // sum_j sU[m, j] B[n, j]
    for (int o = threadIdx.x; o < 16 * M; o += C::THREADS) {
        const int rr = o & 15;
        const int m = o >> 4;
        const int64_t n = n0 + rr;
        if (n >= N) continue;
        float y = red[0][rr][m];
        y += red[1][rr][m];
        y += red[2][rr][m];
        y += red[3][rr][m];
        float l = 0.0f;
        for (int jj = 0; jj < r; ++jj)
            l = fmaf(bf16lo_to_f32(sU[(int64_t)m * ldu + jj]), bf16lo_to_f32(B[n * r + jj]), l);
        Y[(int64_t)m * N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(y + l));
    }
}

}  // namespace qlora
