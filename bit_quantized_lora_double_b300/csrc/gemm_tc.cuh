// gemm_tc.cuh -- fused NF4-dequant + LoRA GEMM on the 5th-generation tensor
// cores (tcgen05, accumulator in TMEM) for sm_103a.
//
//   forward (kFwd):  Y [M, N]  = X [M, K]  . W'^T       + (sU) [M, r] . B^T
//   dX      (kDx):   dX [M, K] = dY [M, N] . W'          + (sV) [M, r] . A
//
// One CTA computes a 128 x 256 tile of the output with BK = 64 per k-step:
//   warp 0       TMA producer: activation tile (128 x 64 bf16, 128-byte
//                swizzle) and the packed-code tile of W (4-bit, 8 KB) per
//                stage; in the LoRA steps the (s*U | s*V) tile and the adapter
//                tile (B or A) instead.
//   warp 1       allocates 256 TMEM columns; one lane issues tcgen05.mma
//                (M = 128, N = 256, K = 16) and commits to mbarriers.
//   warps 2..9   decode the codes of their stage through the per-block scaled
//                byte-plane table straight into the UMMA operand layout
//                (forward: K-major rows of W'; dX: MN-major, k contiguous),
//                fence the generic->async proxy and arrive; after the last
//                k-step they read the fp32 accumulator from TMEM and store
//                bf16 rows.
// The LoRA term enters as ceil(r/64) extra k-steps into the same
// accumulator: [X | sU] . [W' | B]^T and [dY | sV] . [W' ; A].
// Every mbarrier wait is bounded by a time limit; on running out the kernel
// records an error word, stops issuing, drains what it issued and exits.
// Sources: ashishsrivastav.com "QLoRA: Fine-Tuning a 70B on One GPU", section
// "Double Quantization" (dequantize on the fly for the matmul);
// xingyuzhitong.com "Fine-Tuning Memory Requirements", section "QLoRA: quantize
// the frozen base to 4 bits".
#pragma once

#include "common.cuh"

namespace qlora {

enum { kFwd = 0, kDx = 1 };

// One CTA: 256 output rows (two 128-row sub-tiles sharing each decoded W'
// tile) x 256 output columns; two fp32 accumulators fill the 512 TMEM columns.
struct TcCfg {
    static constexpr int BM = 256, SUB = 128, BN = 256, BK = 64, STAGES = 3;
    static constexpr int W_BYTES = BN * BK * 2;    // 32 KB: W' tile (or adapter tile)
    static constexpr int A_BYTES = SUB * BK * 2;   // 16 KB: one activation sub-tile
    static constexpr int C_BYTES = BN * BK / 2;    // 8 KB: packed codes
    static constexpr int STAGE_BYTES = W_BYTES + 2 * A_BYTES + C_BYTES;
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + BAR_BYTES + 1024;
    static constexpr int THREADS = 320;
    static constexpr int DEQ_WARPS = 8;
    static constexpr uint32_t TMEM_COLS = 512;
};

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

template <int MODE>
__global__ void __launch_bounds__(TcCfg::THREADS, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tm_act, const __grid_constant__ CUtensorMap tm_codes,
              const __grid_constant__ CUtensorMap tm_lact, const __grid_constant__ CUtensorMap tm_lw,
              const TcParams p) {
    using C = TcCfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t *full = bar;                       // TMA bytes landed (producer arrive + tx)
    uint64_t *wfull = bar + C::STAGES;          // W' tile decoded (8 warp arrivals)
    uint64_t *empty = bar + 2 * C::STAGES;      // stage consumed by the MMAs (commit)
    uint64_t *accfull = bar + 3 * C::STAGES;    // accumulators complete (commit)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 3 * C::STAGES + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    auto wtile = [&](int s) { return smem + s * C::STAGE_BYTES; };
    auto atile = [&](int s, int h) { return smem + s * C::STAGE_BYTES + C::W_BYTES + h * C::A_BYTES; };
    auto ctile = [&](int s) { return smem + s * C::STAGE_BYTES + C::W_BYTES + 2 * C::A_BYTES; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t m0 = (int64_t)blockIdx.y * C::BM;
    const int64_t c0 = (int64_t)blockIdx.x * C::BN;  // first output column
    // this CTA's share of the contraction: main k-steps [kbeg, kbeg + nmain),
    // then the LoRA steps if it holds the last split
    const int z = (int)blockIdx.z;
    const int64_t kbeg = (int64_t)z * p.steps_per_split;
    const int64_t nmain = max((int64_t)0, min(p.steps_per_split, p.nk_main - kbeg));
    const int64_t nk = nmain + (z == p.splits - 1 ? p.lora_steps : 0);
    const bool two = m0 + C::SUB < p.M;               // second 128-row sub-tile has rows

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&wfull[s], C::DEQ_WARPS);
            mbar_init(&empty[s], 1);
        }
        mbar_init(accfull, 1);
        *abort_flag = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_act);
        prefetch_tmap(&tm_codes);
        prefetch_tmap(&tm_lact);
        prefetch_tmap(&tm_lw);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer ----
        if (lane == 0) {
            const uint32_t abytes = (two ? 2 : 1) * C::A_BYTES;
            int64_t issued = 0;
            for (int64_t it = 0; it < nk; ++it) {
                const int s = (int)(it % C::STAGES);
                const uint32_t u = (uint32_t)(it / C::STAGES);
                if (u > 0 && !tc_wait(&empty[s], (u - 1) & 1, p.wait_ns, (p.kernel_id << 16) | 1, abort_flag)) break;
                if (it < nmain) {
                    mbar_arrive_expect_tx(&full[s], abytes + C::C_BYTES);
                    const int32_t k = (int32_t)((kbeg + it) * C::BK);
                    tma_load_2d(atile(s, 0), &tm_act, &full[s], k, (int32_t)m0);
                    if (two) tma_load_2d(atile(s, 1), &tm_act, &full[s], k, (int32_t)(m0 + C::SUB));
                    if (MODE == kFwd)
                        tma_load_2d(ctile(s), &tm_codes, &full[s], k / 2, (int32_t)c0);
                    else
                        tma_load_2d(ctile(s), &tm_codes, &full[s], (int32_t)(c0 / 2), k);
                } else {
                    const int32_t j = (int32_t)(it - nmain) * C::BK;
                    mbar_arrive_expect_tx(&full[s], abytes + C::W_BYTES);
                    tma_load_2d(atile(s, 0), &tm_lact, &full[s], j, (int32_t)m0);
                    if (two) tma_load_2d(atile(s, 1), &tm_lact, &full[s], j, (int32_t)(m0 + C::SUB));
                    if (MODE == kFwd) {
                        tma_load_2d(wtile(s), &tm_lw, &full[s], j, (int32_t)c0);
                    } else {
#pragma unroll
                        for (int b = 0; b < 4; ++b)
                            tma_load_2d(wtile(s) + b * 8192, &tm_lw, &full[s], (int32_t)(c0 + 64 * b), j);
                    }
                }
                ++issued;
            }
            // drain: the last load issued into each stage must have landed
            for (int s = 0; s < C::STAGES; ++s) {
                if (issued <= s) break;
                const int64_t last = issued - 1 - ((issued - 1 - s) % C::STAGES);
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(&full[s], (uint32_t)(last / C::STAGES) & 1))
                    if (globaltimer() - t0 > p.wait_ns) break;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer ----
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(C::SUB, C::BN, 0, MODE == kDx ? 1 : 0);
            for (int64_t it = 0; it < nk; ++it) {
                const int s = (int)(it % C::STAGES);
                const uint32_t par = (uint32_t)(it / C::STAGES) & 1;
                if (!tc_wait(&full[s], par, p.wait_ns, (p.kernel_id << 16) | 3, abort_flag)) break;
                if (!tc_wait(&wfull[s], par, p.wait_ns, (p.kernel_id << 16) | 4, abort_flag)) break;
                tc_fence_after();
                int nmma = 4;
                if (it >= nmain) {
                    const int rem = p.r - (int)(it - nmain) * C::BK;
                    nmma = rem >= C::BK ? 4 : (rem + 15) / 16;
                }
                const uint32_t a0 = smem_u32(atile(s, 0)), a1 = smem_u32(atile(s, 1)), w0 = smem_u32(wtile(s));
                for (int kk = 0; kk < nmma; ++kk) {
                    const uint64_t bd = MODE == kFwd ? smem_desc_sw128(w0 + kk * 32, 16, 1024)
                                                     : smem_desc_sw128(w0 + kk * 2048, 8192, 1024);
                    const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
                    tc_mma_bf16(tmem, smem_desc_sw128(a0 + kk * 32, 16, 1024), bd, idesc, acc);
                    if (two) tc_mma_bf16(tmem + 256, smem_desc_sw128(a1 + kk * 32, 16, 1024), bd, idesc, acc);
                }
                tc_commit(&empty[s]);
            }
            tc_commit(accfull);
        }
    } else {
        // ------------------------------------- decode, then epilogue ----
        const int dt = threadIdx.x - 64;  // 0..255
        const float mean = *p.mean;
        const int64_t kblocks = p.w_cols / kBlock;
        // This thread's W row / 64-column block at k-step `it`, its slot in
        // the code tile and the byte offsets of its 8 output chunks.
        int64_t wrow0, kb0, wrow_step, kb_step;
        int crow, ccol;
        uint32_t dst[8];
        if (MODE == kFwd) {
            // row c0 + dt of W, block `it`; K-major 128-byte swizzled row
            wrow0 = c0 + dt;
            wrow_step = 0;
            kb0 = 0;
            kb_step = 1;
            crow = dt;
            ccol = 0;
#pragma unroll
            for (int c = 0; c < 8; ++c) dst[c] = (uint32_t)((dt >> 3) * 1024 + (dt & 7) * 128 + ((c ^ (dt & 7)) << 4));
        } else {
            // row it*64 + nl of W (K-group of the MN-major operand), block b4
            const int nlo = dt & 7, b4 = (dt >> 3) & 3, nhi = dt >> 5;
            const int nl = nhi * 8 + nlo;
            wrow0 = nl;
            wrow_step = C::BK;
            kb0 = c0 / kBlock + b4;
            kb_step = 0;
            crow = nl;
            ccol = b4;
#pragma unroll
            for (int c = 0; c < 8; ++c) dst[c] = (uint32_t)(b4 * 8192 + nhi * 1024 + nlo * 128 + ((c ^ nlo) << 4));
        }
        // absmax code and scale for local k-step `it` (prefetched one step ahead)
        auto fetch = [&](int64_t it, int &qv, float &sv) {
            const int64_t g = kbeg + it;
            const int64_t wrow = wrow0 + g * wrow_step, kb = kb0 + g * kb_step;
            if (it < nmain && wrow < p.w_rows && kb < kblocks) {
                const int64_t b = wrow * kblocks + kb;
                qv = __ldg(p.q + b);
                sv = __ldg(p.s2 + (b >> 8));
                return true;
            }
            qv = 0;
            sv = 0.0f;
            return false;
        };
        int q_cur, q_nxt;
        float s_cur, s_nxt;
        bool v_cur = fetch(0, q_cur, s_cur), v_nxt = false;
        bool alive = true;
        for (int64_t it = 0; it < nk && alive; ++it) {
            const int s = (int)(it % C::STAGES);
            const uint32_t par = (uint32_t)(it / C::STAGES) & 1;
            v_nxt = fetch(it + 1, q_nxt, s_nxt);
            if (!tc_wait(&full[s], par, p.wait_ns, (p.kernel_id << 16) | 2, abort_flag)) {
                alive = false;
                break;
            }
            if (it < nmain) {
                uint8_t *wt = wtile(s);
                const uint8_t *ct = ctile(s);
                uint32_t o[8][4];
                if (v_cur) {
                    const Nf4Table tab = make_table(dq_absmax((int8_t)q_cur, s_cur, mean));
                    uint4 cw[2];
                    if (MODE == kFwd) {
                        // 32-byte rows, 32-byte swizzle: half h sits at h ^ bit 2 of the row
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            cw[h] = *reinterpret_cast<const uint4 *>(ct + crow * 32 + ((h ^ ((crow >> 2) & 1)) << 4));
                    } else {
                        // 128-byte rows, 128-byte swizzle
#pragma unroll
                        for (int h = 0; h < 2; ++h)
                            cw[h] = *reinterpret_cast<const uint4 *>(ct + crow * 128 + (((ccol * 2 + h) ^ (crow & 7)) << 4));
                    }
                    const uint32_t w[8] = {cw[0].x, cw[0].y, cw[0].z, cw[0].w, cw[1].x, cw[1].y, cw[1].z, cw[1].w};
#pragma unroll
                    for (int c = 0; c < 8; ++c) decode8(tab, w[c], o[c]);
                } else {
#pragma unroll
                    for (int c = 0; c < 8; ++c) o[c][0] = o[c][1] = o[c][2] = o[c][3] = 0u;
                }
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4 *>(wt + dst[c]) = make_uint4(o[c][0], o[c][1], o[c][2], o[c][3]);
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&wfull[s]);
            q_cur = q_nxt;
            s_cur = s_nxt;
            v_cur = v_nxt;
        }
        // ------------------------------------------------------ epilogue
        const bool acc_ok = tc_wait(accfull, 0, p.wait_ns, (p.kernel_id << 16) | 5, abort_flag);
        tc_fence_after();
        const int quarter = warp & 3, sub = (warp - 2) >> 2;
        if (acc_ok && alive && (sub == 0 || two)) {
            const int64_t row = m0 + sub * C::SUB + quarter * 32 + lane;
#pragma unroll 1
            for (int cc = 0; cc < C::BN / 32; ++cc) {
                const int col = cc * 32;
                uint32_t v[32];
                tmem_ld_32x32b_x32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(sub * 256 + col), v);
                tmem_ld_wait();
                const int64_t ncol = p.Nd - (c0 + col);  // valid columns from here
                if (row < p.M && p.splits > 1) {
                    float *dstf = p.part + ((int64_t)z * p.M + row) * p.Nd + c0 + col;
                    if (ncol >= 32 && ((p.Nd & 3) == 0)) {
#pragma unroll
                        for (int g = 0; g < 8; ++g)
                            reinterpret_cast<float4 *>(dstf)[g] =
                                make_float4(__uint_as_float(v[4 * g]), __uint_as_float(v[4 * g + 1]),
                                            __uint_as_float(v[4 * g + 2]), __uint_as_float(v[4 * g + 3]));
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (e < ncol) dstf[e] = __uint_as_float(v[e]);
                    }
                } else if (row < p.M) {
                    uint16_t *dstp = p.out + row * p.ldo + c0 + col;
                    if (ncol >= 32 && ((p.ldo & 7) == 0)) {
#pragma unroll
                        for (int g = 0; g < 4; ++g) {
                            uint4 pk;
                            pk.x = pack_bf16x2(__uint_as_float(v[8 * g + 0]), __uint_as_float(v[8 * g + 1]));
                            pk.y = pack_bf16x2(__uint_as_float(v[8 * g + 2]), __uint_as_float(v[8 * g + 3]));
                            pk.z = pack_bf16x2(__uint_as_float(v[8 * g + 4]), __uint_as_float(v[8 * g + 5]));
                            pk.w = pack_bf16x2(__uint_as_float(v[8 * g + 6]), __uint_as_float(v[8 * g + 7]));
                            reinterpret_cast<uint4 *>(dstp)[g] = pk;
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (e < ncol) dstp[e] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[e])));
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

}  // namespace qlora

namespace qlora {

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
