// lora_tc.cuh -- the LoRA side path on the tensor cores: skinny GEMMs whose
// output has at most 64 columns per tile (the rank) and whose contraction is
// long (K, N or the M tokens).
//
//   U    = X  A^T     out [M, r]   A-op X  [M, K]  K-major, B-op A  [r, K] K-major
//   V    = dY B       out [M, r]   A-op dY [M, N]  K-major, B-op B  [N, r] MN-major
//   dA^T = X^T (sV)   out [K, r]   A-op X  [M, K]  MN-major, B-op sV [M, r] MN-major
//   dB   = dY^T U     out [N, r]   A-op dY [M, N]  MN-major, B-op U  [M, r] MN-major
//
// Grid: (128-row output tiles, contraction chunks, 64-wide rank tiles); the
// chunks of one tile form one thread-block cluster (at most 8 CTAs). Each
// CTA streams its chunk through an 8-stage TMA pipeline (192 KB in flight) and
// accumulates a 128 x 64 fp32 tile in TMEM with tcgen05.mma (M=128, N=64,
// K=16). The rank is padded to 64 by the TMA's zero fill of out-of-range
// elements, so no padded copy of A, B or U is needed when r % 8 == 0.
// Every CTA of a cluster leaves its fp32 partial tile in its own shared
// memory; after a cluster barrier the first CTA adds the partials over
// distributed shared memory in chunk order (a fixed order) and writes the
// outputs; a second cluster barrier keeps the partials alive until then.
// Sources: xingyuzhitong.com "Fine-Tuning Memory Requirements: Full Training vs
// LoRA vs QLoRA", section "LoRA: freeze the base, train small adapters";
// inquiringlines.com note, mechanism paragraph (gradients flow only into the
// adapters).
#pragma once

#include "common.cuh"
#include "gemm_tc.cuh"

namespace qlora {

// Output written by the tile reduction.
//   kRedU:  U [rows, lda] bf16 = sum (if o16a), sU [rows, ldb] bf16 = bf16(s * sum)
//   kRedV:  sV [rows, ldb] bf16 = bf16(s * sum)
//   kRedDA: dA [r, rows] fp32 = sum (element [j, row])
//   kRedDB: dB [rows, r] fp32 = s * sum
// For kRedU and kRedV, columns [r, zend) of sU / sV are written as zeros
// (zend <= ldb).
enum { kRedU = 0, kRedV = 1, kRedDA = 2, kRedDB = 3 };

#ifndef QLORA_SK_STAGES
#define QLORA_SK_STAGES 8
#endif
#ifndef QLORA_SK_MIN_BLOCKS
#define QLORA_SK_MIN_BLOCKS 1
#endif

struct SkCfg {
    static constexpr int BM = 128, BN = 64, BK = 64, STAGES = QLORA_SK_STAGES;
    static constexpr int A_BYTES = BM * BK * 2;  // 16 KB
    static constexpr int B_BYTES = BN * BK * 2;  // 8 KB
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 256 + 1024;
    static constexpr int THREADS = 192;
    static constexpr uint32_t TMEM_COLS = 64;
};

struct SkParams {
    int64_t rows;             // valid output rows
    int64_t L;                // contraction length
    int64_t steps_per_chunk;  // 64-deep steps per chunk
    int nchunks;              // chunks per tile = cluster size along y
    int r;                    // valid output columns (the rank)
    float s;                  // LoRA scale
    int mode;                 // kRed*
    uint16_t *o16a;
    int lda;
    uint16_t *o16b;
    int ldb;
    int zend;
    float *o32;
    uint64_t wait_ns;
    unsigned kernel_id;
    uint32_t *zero;  // problem 0 only: words set to zero once the preceding kernel is done
    int nzero;
};

// floats per row of the partial tile kept in shared memory (64 + 4 padding:
// rows 16 bytes apart in bank terms, so a quarter-warp's float4 accesses to
// 8 consecutive rows hit distinct banks)
constexpr int kRedStride = 68;
// largest cluster (chunks of one tile's contraction) the host plans
constexpr int kSkMaxCluster = 8;

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(saddr), "r"(rank));
    return d;
}
__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}
// All threads of all CTAs of the cluster (a cluster of one CTA is a plain
// CTA-wide barrier).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Writes row `row`, rank columns jbase .. jbase + 63 (those below r) of the
// tile's complete sum.
__device__ __forceinline__ void sk_store(const SkParams &p, int64_t row, int jbase, const float (&acc)[64]) {
    const int nj = min(64, p.r - jbase);
    const bool last_z = jbase + 64 >= p.r;
    switch (p.mode) {
        case kRedU:
        case kRedV: {
            uint16_t *ob = p.o16b + row * p.ldb + jbase;
#pragma unroll
            for (int j = 0; j < 64; ++j) {
                if (j < nj) {
                    if (p.mode == kRedU && p.o16a)
                        p.o16a[row * p.lda + jbase + j] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[j]));
                    ob[j] = __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(p.s, acc[j])));
                }
            }
            if (last_z)
                for (int jj = p.r; jj < p.zend; ++jj) p.o16b[row * p.ldb + jj] = 0;
            break;
        }
        case kRedDA:
#pragma unroll
            for (int j = 0; j < 64; ++j)
                if (j < nj) p.o32[(int64_t)(jbase + j) * p.rows + row] = acc[j];
            break;
        default:
#pragma unroll
            for (int j = 0; j < 64; ++j)
                if (j < nj) p.o32[row * p.r + jbase + j] = __fmul_rn(p.s, acc[j]);
            break;
    }
}

// Writes row `row`, columns j0 .. j0 + nv - 1 (nv <= 4) of the tile's
// complete sum, v holding those values in order; `pad` also writes the zero
// columns [r, zend) of sU / sV for that row.
__device__ __forceinline__ void sk_store4(const SkParams &p, int64_t row, int j0, int nv, float4 v, bool pad) {
    const float a[4] = {v.x, v.y, v.z, v.w};
    switch (p.mode) {
        case kRedU:
        case kRedV: {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (e < nv) {
                    if (p.mode == kRedU && p.o16a)
                        p.o16a[row * p.lda + j0 + e] = __bfloat16_as_ushort(__float2bfloat16_rn(a[e]));
                    p.o16b[row * p.ldb + j0 + e] = __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(p.s, a[e])));
                }
            }
            if (pad)
                for (int jj = p.r; jj < p.zend; ++jj) p.o16b[row * p.ldb + jj] = 0;
            break;
        }
        case kRedDA:
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (e < nv) p.o32[(int64_t)(j0 + e) * p.rows + row] = a[e];
            break;
        default:
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (e < nv) p.o32[row * p.r + j0 + e] = __fmul_rn(p.s, a[e]);
            break;
    }
}

// One launch carries up to kSkMaxJobs problems of the same kind (the same
// operand majorness) and rank-tile count: CTAs with first[j] <= blockIdx.x <
// first[j + 1] take problem j (maps a[j], b[j]). The problems share the
// cluster size (contraction chunks per tile); each splits its own contraction
// into that many chunks (chunks past its end stream nothing and add zeros).
constexpr int kSkMaxJobs = 5;
struct SkMaps {
    CUtensorMap a[kSkMaxJobs];
    CUtensorMap b[kSkMaxJobs];
};
struct SkBatch {
    SkParams p[kSkMaxJobs];
    int first[kSkMaxJobs + 1];
    int n;
};

template <int A_MN, int B_MN>
__global__ void __launch_bounds__(SkCfg::THREADS, QLORA_SK_MIN_BLOCKS)
    k_lora_skinny(const __grid_constant__ SkMaps tm, const __grid_constant__ SkBatch bt) {
    using C = SkCfg;
    int job = 0;
    while (job + 1 < bt.n && (int)blockIdx.x >= bt.first[job + 1]) ++job;
    const SkParams &p = bt.p[job];
    const CUtensorMap *tm_a = &tm.a[job];
    const CUtensorMap *tm_b = &tm.b[job];
    const int64_t tile = (int64_t)blockIdx.x - bt.first[job];
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t *full = bar, *empty = bar + C::STAGES, *accfull = bar + 2 * C::STAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 2 * C::STAGES + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    auto atile = [&](int s) { return smem + s * C::STAGE_BYTES; };
    auto btile = [&](int s) { return smem + s * C::STAGE_BYTES + C::A_BYTES; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row0 = tile * C::BM;
    const int64_t l0 = (int64_t)blockIdx.y * p.steps_per_chunk * C::BK;
    int64_t nsteps = (p.L - l0 + C::BK - 1) / C::BK;
    if (nsteps > p.steps_per_chunk) nsteps = p.steps_per_chunk;
    if (nsteps < 0) nsteps = 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(accfull, 1);
        *abort_flag = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(tm_a);
        prefetch_tmap(tm_b);
        // the first stages' streamed tiles into L2 while the preceding kernel
        // finishes (L2 stays coherent with its writes)
        for (int64_t it = 0; it < nsteps && it < 4; ++it) {
            const int32_t l = (int32_t)(l0 + it * C::BK);
            if (A_MN) {
                tma_prefetch_2d(tm_a, (int32_t)row0, l);
                tma_prefetch_2d(tm_a, (int32_t)(row0 + 64), l);
            } else {
                tma_prefetch_2d(tm_a, l, (int32_t)row0);
            }
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // launched as a programmatic dependent of the preceding kernel: its
    // outputs are visible from here on; the next kernel may start its set-up
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (bt.p[0].zero && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
        for (int i = threadIdx.x; i < bt.p[0].nzero; i += blockDim.x) bt.p[0].zero[i] = 0u;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer ----
        if (lane == 0) {
            int64_t issued = 0;
            const int32_t jz = (int32_t)blockIdx.z * C::BN;
            for (int64_t it = 0; it < nsteps; ++it) {
                const int s = (int)(it % C::STAGES);
                const uint32_t u = (uint32_t)(it / C::STAGES);
                if (u > 0 && !tc_wait(&empty[s], (u - 1) & 1, p.wait_ns, (p.kernel_id << 16) | 1, abort_flag)) break;
                const int32_t l = (int32_t)(l0 + it * C::BK);
                mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
                if (A_MN) {
                    tma_load_2d(atile(s), tm_a, &full[s], (int32_t)row0, l);
                    tma_load_2d(atile(s) + 8192, tm_a, &full[s], (int32_t)(row0 + 64), l);
                } else {
                    tma_load_2d(atile(s), tm_a, &full[s], l, (int32_t)row0);
                }
                if (B_MN)
                    tma_load_2d(btile(s), tm_b, &full[s], jz, l);
                else
                    tma_load_2d(btile(s), tm_b, &full[s], l, jz);
                ++issued;
            }
            // drain: the last load issued into each stage must have landed
            for (int s = 0; s < C::STAGES; ++s) {
                if (issued <= s) break;
                const int64_t last = issued - 1 - ((issued - 1 - s) % C::STAGES);
                drain_wait(&full[s], (uint32_t)(last / C::STAGES) & 1);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer ----
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(C::BM, C::BN, A_MN, B_MN);
            for (int64_t it = 0; it < nsteps; ++it) {
                const int s = (int)(it % C::STAGES);
                if (!tc_wait(&full[s], (uint32_t)(it / C::STAGES) & 1, p.wait_ns, (p.kernel_id << 16) | 3, abort_flag))
                    break;
                tc_fence_after();
                const uint32_t a0 = smem_u32(atile(s)), b0 = smem_u32(btile(s));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t ad = A_MN ? smem_desc_sw128(a0 + kk * 2048, 8192, 1024)
                                             : smem_desc_sw128(a0 + kk * 32, 16, 1024);
                    const uint64_t bd = B_MN ? smem_desc_sw128(b0 + kk * 2048, 8192, 1024)
                                             : smem_desc_sw128(b0 + kk * 32, 16, 1024);
                    tc_mma_bf16(tmem, ad, bd, idesc, (it > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(&empty[s]);
            }
            tc_commit(accfull);
            // every MMA issued has completed before TMEM is given up (after an
            // abort the epilogue does not wait for this commit)
            drain_wait(accfull, 0);
        }
    } else {
        // -------------------- warps 2..5: one output row per thread ----
        const bool ok = tc_wait(accfull, 0, p.wait_ns, (p.kernel_id << 16) | 5, abort_flag);
        tc_fence_after();
        const int quarter = warp & 3;  // TMEM lanes this warp may read
        const int trow = quarter * 32 + lane;
        const int64_t row = row0 + trow;
        const int jbase = (int)blockIdx.z * C::BN;
        const int nj = min(64, p.r - jbase);
        float acc[64];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(h * 32), v);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) acc[h * 32 + e] = (ok && nsteps > 0) ? __uint_as_float(v[e]) : 0.0f;
        }
        if (p.nchunks == 1) {
            if (ok && row < p.rows) sk_store(p, row, jbase, acc);
        } else {
            // the partial tile goes to this CTA's shared memory (the stage
            // buffers: every load has landed and been consumed by now)
            float *red = reinterpret_cast<float *>(smem) + trow * kRedStride;
#pragma unroll
            for (int g = 0; g < 16; ++g)
                if (4 * g < nj)
                    reinterpret_cast<float4 *>(red)[g] = make_float4(acc[4 * g], acc[4 * g + 1], acc[4 * g + 2],
                                                                     acc[4 * g + 3]);
        }
    }
    tc_fence_before();
    __syncwarp();
    if (p.nchunks > 1) {
        cluster_sync_all();  // every partial tile of the cluster is in place
        if (warp >= 2) {
            // The cluster's CTAs share the reduction: work item u covers tile
            // row u % BM, columns 4 * (u / BM) .. + 3 of this z-slice, and
            // sums that float4 over the n partial tiles (c = 0 .. n - 1, in
            // that order). Items are dealt out over the 128 epilogue threads
            // of every CTA, so all n remote loads of an item are in flight
            // together and no CTA walks the whole tile.
            const int n = p.nchunks;  // <= kSkMaxCluster
            const int jbase = (int)blockIdx.z * C::BN;
            const int nj = min(64, p.r - jbase);
            const int ng = (nj + 3) >> 2;
            const bool last_z = jbase + 64 >= p.r;
            const uint32_t local = smem_u32(smem);
            uint32_t base[kSkMaxCluster];
#pragma unroll
            for (int c = 0; c < kSkMaxCluster; ++c) base[c] = c < n ? mapa_shared(local, (uint32_t)c) : 0u;
            const int stride = n * C::BM;
            for (int u = (int)cluster_ctarank() * C::BM + ((int)threadIdx.x - 64); u < C::BM * ng; u += stride) {
                const int trow = u % C::BM, g = u / C::BM;
                const int64_t row = row0 + trow;
                if (row >= p.rows) continue;
                const uint32_t off = (uint32_t)(trow * kRedStride + 4 * g) * 4u;
                float4 f[kSkMaxCluster];
#pragma unroll
                for (int c = 0; c < kSkMaxCluster; ++c)
                    if (c < n) f[c] = ld_dsmem_f4(base[c] + off);
                float4 sum = f[0];
#pragma unroll
                for (int c = 1; c < kSkMaxCluster; ++c) {
                    if (c < n) {
                        sum.x += f[c].x;
                        sum.y += f[c].y;
                        sum.z += f[c].z;
                        sum.w += f[c].w;
                    }
                }
                sk_store4(p, row, jbase + 4 * g, min(4, nj - 4 * g), sum, last_z && g == ng - 1);
            }
        }
        __syncwarp();
        // the partials stay alive until every remote read has returned (the
        // sums are already stored: no ordering of memory needed here)
        asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

}  // namespace qlora
