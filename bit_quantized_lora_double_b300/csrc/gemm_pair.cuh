// gemm_pair.cuh -- fused NF4-dequant + LoRA GEMM on a CTA pair (tcgen05
// cta_group::2) for sm_103a.
//
//   forward (kFwd):  Y [M, N]  = X [M, K]  . W'^T       + (sU) [M, r] . B^T
//   dX      (kDx):   dX [M, K] = dY [M, N] . W'          + (sV) [M, r] . A
//
// Two CTAs of a cluster compute a 512 x 256 output tile together. Each
// tcgen05.mma (M = 256, N = 256, K = 16) issued by the even CTA reads 128
// activation rows and 128 of the 256 weight columns from each CTA's shared
// memory and accumulates 128 x 256 fp32 in each CTA's TMEM. Two such 256-row
// sub-tiles fill the 512 TMEM columns, so every decoded weight tile feeds
// 2 x 256 rows while each CTA decodes only its half of it: 128 x 64 weights
// per 64-deep k-step against 2 x (128 x 256 x 64) MACs.
//
// Roles per CTA (14 warps):
//   warp 0      TMA producer: two 128 x 64 activation tiles and this CTA's
//               half of the packed-code tile per stage (in the LoRA steps
//               the s*U or s*V tiles and this CTA's half of the adapter
//               tile instead).
//   warp 1      TMEM allocation (both CTAs); in the even CTA one lane waits
//               until both halves of a stage are decoded, issues the MMAs and
//               commits to the stage's `empty` barriers of both CTAs.
//   warps 2..9  two decode groups of 4 warps taking alternate k-steps: each
//               thread expands one block of 64 codes through the per-block
//               scaled byte-plane table into the UMMA operand layout, then
//               arrives on the even CTA's `ready` barrier.
//   warps 10..13 the epilogue, one warp per TMEM lane quarter: accumulators
//               to bf16 output rows (or to a stream-K partial slot).
// The LoRA term enters as ceil(r/64) extra k-steps into the same
// accumulators. Every wait is bounded in time; a wait that runs out records
// the error word, raises the abort flag in both CTAs, and the kernel drains
// and exits.
// Sources: ashishsrivastav.com "QLoRA: Fine-Tuning a 70B on One GPU", section
// "Double Quantization" (dequantize on the fly for the matmul);
// xingyuzhitong.com "Fine-Tuning Memory Requirements", section "QLoRA: quantize
// the frozen base to 4 bits".
#pragma once

#include "common.cuh"
#include "gemm_tc.cuh"

namespace qlora {

// Diagnostic timeline (built only with -DQLORA_GEMM_STAMPS, into a separate
// library): globaltimer stamps of the first CTA pair of the last launch, per
// k-step g (rows 0-4, 7) or per tile (rows 5, 6):
//   0 producer: stage free, loads about to be issued     (CTA 0)
//   1 decode group: the stage's bytes have landed          (CTA 0, first warp)
//   2 decode group: decoded tile stored                    (CTA 0, first warp)
//   3 MMA issuer: decoded halves ready                     (CTA 0)
//   4 MMA issuer: MMAs issued and committed                (CTA 0)
//   5 epilogue: accumulators complete                      (CTA 0, warp 0)
//   6 epilogue: accumulators read, released to the MMAs    (CTA 0, warp 0)
//   7 decode group: decoded tile stored                    (CTA 1, first warp)
#ifdef QLORA_GEMM_STAMPS
constexpr int kStampSteps = 4096;
__device__ unsigned long long d_gemm_stamps[8][kStampSteps];
#define QLORA_STAMP(row, cta, idx)                                                                    \
    do {                                                                                              \
        if (blockIdx.x == (cta) && (idx) < kStampSteps) d_gemm_stamps[row][idx] = globaltimer();        \
    } while (0)
#else
#define QLORA_STAMP(row, cta, idx) \
    do {                           \
    } while (0)
#endif

struct PairCfg {
    static constexpr int SUB = 128;               // rows per CTA per sub-tile
    static constexpr int PAIR_M = 512;            // rows per pair tile (2 sub-tiles x 256)
    static constexpr int BN = 256, HN = 128, BK = 64, STAGES = 4;
    static constexpr int A_BYTES = SUB * BK * 2;  // 16 KB: one activation tile
    static constexpr int W_BYTES = HN * BK * 2;   // 16 KB: this CTA's half of W' (or adapter)
    static constexpr int C_BYTES = HN * BK / 2;   // 4 KB: this CTA's half of the codes
    static constexpr int STAGE_BYTES = W_BYTES + 2 * A_BYTES + C_BYTES;
    static constexpr int BAR_BYTES = 512;
    static constexpr int NFIX = 6;                // 8 KB partial pieces in flight per epilogue warp when finishing
    static constexpr int GROUP_WARPS = 4;         // decode warps per group
    static constexpr int DEC_GROUPS = 2;          // groups take alternate k-steps
    static constexpr int EPI_WARPS = 4;           // one per TMEM lane quarter
    // per epilogue warp: 4 KB output staging, 1 KB aligned (128-byte swizzle)
    static constexpr int EPI_OFF = STAGES * STAGE_BYTES + 1024;
    static constexpr int SMEM_BYTES = EPI_OFF + 4 * 4096 + 1024;
    static constexpr int NBATCH = 8;              // 64-column batches per warp and tile (2 sub-tiles x 4)
    static constexpr int THREADS = 64 + 32 * (GROUP_WARPS * DEC_GROUPS + EPI_WARPS);
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int MAX_PAIRS = 74;
};
static_assert(PairCfg::MAX_PAIRS == kSkPairs, "one stream-K slot and flag set per pair");
static_assert(PairCfg::SMEM_BYTES <= 232448, "shared memory per CTA");
static_assert(PairCfg::BAR_BYTES <= 1024 && PairCfg::EPI_OFF % 1024 == 0, "barriers before the staging tiles");
static_assert(PairCfg::EPI_WARPS * PairCfg::NFIX * 8192 <= PairCfg::STAGES * PairCfg::STAGE_BYTES,
              "finishing buffers live in the stage ring");

// ---- cta_group::2 wrappers -------------------------------------------------
__device__ __forceinline__ void tmem_alloc2(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_mma2_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on the barrier at this shared-memory offset in every CTA of
// the pair when all tcgen05 operations issued so far by this thread complete.
__device__ __forceinline__ void tc_commit2_both(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"((uint16_t)0x3)
        : "memory");
}
// Arrive once on this CTA's barrier `bar` when all tcgen05 operations issued
// so far by this thread complete.
__device__ __forceinline__ void tc_commit2_self(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ uint32_t pair_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r & 1u;
}
__device__ __forceinline__ uint32_t mapa_u32(uint32_t saddr, uint32_t rank) {
    uint32_t d;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(d) : "r"(saddr), "r"(rank));
    return d;
}
// Arrive (release, cluster scope) on an mbarrier given by its shared::cluster
// address (possibly in the peer CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
__device__ __forceinline__ void pair_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 32-byte global store (address 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void *p, const uint32_t (&v)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v[0]), "r"(v[1]),
                 "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}
// Programmatic dependent launch: wait for the preceding kernel's memory, and
// let the next kernel start its own set-up.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// Bounded wait like tc_wait; on running out it also raises the peer CTA's
// abort flag (given by its shared::cluster address).
__device__ __forceinline__ bool pair_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns, unsigned code,
                                          volatile int *abort_flag, uint32_t peer_abort) {
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
            st_cluster_u32(peer_abort, 1u);
            return false;
        }
    }
}

// Work schedule: data-parallel waves, then a stream-K remainder. The T
// output tiles of 512 x 256 are numbered band by band (p.band row tiles per
// band), with the row tiles of a column tile adjacent inside a band; each is
// S = nk_main + lora_steps k-steps deep. Tiles t < dp_tiles
// go data-parallel: pair q of the P pairs computes tiles q, q + P, ... whole,
// all pairs in step (neighbouring pairs share weight and activation tiles
// through L2 at the same k). The remaining tiles form one line of
// W = (T - dp_tiles) * S steps, and pair q takes steps [q W / P, (q + 1) W / P)
// of it. Inside that range a pair works through segments, one per tile
// touched:
//   kSegFull  the whole tile: the pair writes the output;
//   kSegPart  a later part of the tile (the range starts inside the tile):
//             always the pair's first stream-K segment;
//   kSegHead  the tile's first steps (the range ends inside the tile): always
//             the pair's last segment.
// A shared tile's contributors are its head pair h and the pairs h + 1 ..
// h + n - 1 whose ranges start inside it. Each epilogue warp of each
// contributor, once its accumulators are complete, counts itself in on the
// tile's arrival counter. The last to arrive finishes the tile: it waits for
// the others' ready flags, adds their fp32 partials and its own accumulators
// in pair order (so the sum is the same whoever arrives last) and writes the
// output. Every other contributor writes its partial to its slot (the head
// slot or the tail slot: a pair may hold one of each) and raises the slot's
// ready flag. A pair only ever waits for contributors that have already
// arrived, so no pair depends on another pair being resident or making
// progress. With the host's schedule a shared tile has at most four
// contributors, and the head, whose segment is its pair's last, usually
// arrives last.
enum { kSegFull = 0, kSegHead = 1, kSegPart = 2 };

struct PairSeg {
    int64_t t, m0;
    int64_t c0;     // first output column, within the column group's projection
    int cg;         // column group (forward: the projection)
    int64_t kbeg;   // first main k-step
    int64_t nmain;  // main k-steps
    int64_t lbeg;   // first LoRA k-step
    int64_t nk;     // all k-steps
    int role;
    bool two;       // the tile has a second 256-row sub-tile
};

// Row tiles per band of the tile order (TcParams::band, chosen per launch by
// the host): the pairs working at the same time touch at most this many row
// tiles, so the band's activation rows stay in L2 across the band's
// data-parallel rounds while every column tile passes; a smaller band reads
// each weight column tile once per band instead. The host takes the largest
// band of 8, 4, 2 or 1 row tiles whose activation slice fits kBandBytes.

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

struct PairPlan {
    int64_t mt, nt, S, T, dpt, P;
    int64_t base, W;  // stream-K line: steps [base, base + W)
    __host__ __device__ __forceinline__ int64_t begin(int64_t q) const { return base + W * q / P; }
};

// The schedule of one launch on P pairs (tile_rows and dp_tiles set by the host).
__host__ __device__ __forceinline__ PairPlan make_plan(const TcParams &p, int64_t P) {
    PairPlan pl;
    pl.mt = (p.M + p.tile_rows - 1) / p.tile_rows;
    pl.S = p.nk_main + p.lora_steps;
    pl.nt = (p.Nd + PairCfg::BN - 1) / PairCfg::BN;
    pl.T = pl.mt * pl.nt;
    pl.dpt = min64(p.dp_tiles, pl.T);
    pl.P = P;
    pl.base = pl.dpt * pl.S;
    pl.W = (pl.T - pl.dpt) * pl.S;
    return pl;
}

// The pair finishing tile t (its head, pair q) adds the tails computed by
// pairs q + 1 .. head_contrib_end(...) - 1: those whose ranges start inside t.
__host__ __device__ __forceinline__ int64_t head_contrib_end(const PairPlan &pl, int64_t q, int64_t t) {
    const int64_t tend = (t + 1) * pl.S;
    int64_t e = q + 1;
    while (e < pl.P && pl.begin(e) < tend) ++e;
    return e;
}

// The pair computing tile t's first steps: the last pair whose range begins
// at or before step t * S (pair q's range begins after it).
__host__ __device__ __forceinline__ int64_t head_pair(const PairPlan &pl, int64_t q, int64_t t) {
    int64_t h = q;
    while (h > 0 && pl.begin(h) > t * pl.S) --h;
    return h;
}

// Walks one pair's segments: its data-parallel tiles, then its stream-K range.
struct SegWalk {
    int64_t dp;   // next data-parallel tile
    int64_t g;    // next stream-K step
    int64_t end;  // end of this pair's stream-K range
};

__host__ __device__ __forceinline__ PairSeg pair_seg(const TcParams &p, const PairPlan &pl, int64_t g,
                                                     int64_t end);

__host__ __device__ __forceinline__ SegWalk seg_walk(const PairPlan &pl, int64_t q) {
    SegWalk sw;
    sw.dp = q;
    sw.g = pl.begin(q);
    sw.end = pl.begin(q + 1);
    return sw;
}
__host__ __device__ __forceinline__ bool seg_next(const TcParams &p, const PairPlan &pl, SegWalk &sw, PairSeg &w) {
    if (sw.dp < pl.dpt) {
        w = pair_seg(p, pl, sw.dp * pl.S, sw.dp * pl.S + pl.S);
        sw.dp += pl.P;
        return true;
    }
    if (sw.g < sw.end) {
        w = pair_seg(p, pl, sw.g, sw.end);
        sw.g += w.nk;
        return true;
    }
    return false;
}

__host__ __device__ __forceinline__ PairSeg pair_seg(const TcParams &p, const PairPlan &pl, int64_t g,
                                                     int64_t end) {
    PairSeg w;
    w.t = g / pl.S;
    const int64_t k0 = g - w.t * pl.S, k1 = min64(pl.S, k0 + (end - g));
    // tile t -> (row tile, column tile): bands of p.band row tiles, the
    // row tiles of a column tile adjacent inside a band
    const int64_t rbnd = p.band > 0 ? p.band : 1;
    const int64_t band = w.t / (rbnd * pl.nt);
    const int64_t rows_in = min64(rbnd, pl.mt - band * rbnd);
    const int64_t rb = w.t - band * rbnd * pl.nt;
    w.m0 = (band * rbnd + rb % rows_in) * p.tile_rows;
    const int64_t ct = rb / rows_in;  // column tile of the launch
    int cg = 0;
    while (cg + 1 < p.ncg && ct >= p.cg_first[cg + 1]) ++cg;
    w.cg = cg;
    w.c0 = (ct - p.cg_first[cg]) * PairCfg::BN;
    w.kbeg = k0;
    w.nmain = max64(0, min64(k1, p.nk_main) - k0);
    w.lbeg = max64(k0, p.nk_main) - p.nk_main;
    w.nk = k1 - k0;
    w.role = k0 == 0 ? (k1 == pl.S ? kSegFull : kSegHead) : kSegPart;
    w.two = p.tile_rows == PairCfg::PAIR_M && w.m0 + 256 < p.M;
    return w;
}

// Global -> shared bulk copy completing on an mbarrier of this CTA.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// 16-byte load through a generic address (shared or global memory), at gpu
// scope so a global address never reads a stale L1 line.
__device__ __forceinline__ float4 ld_f4_gpu(const float *p) {
    float4 v;
    asm volatile("ld.relaxed.gpu.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}
__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
// Bounded wait for a ready flag raised by another pair.
__device__ __forceinline__ bool flag_wait(const uint32_t *f, uint64_t limit_ns, unsigned code,
                                          volatile int *abort_flag, uint32_t peer_abort) {
    if (ld_acquire_gpu(f)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
        __nanosleep(256);
        if (ld_acquire_gpu(f)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > limit_ns) {
            record_error(code);
            *abort_flag = 1;
            st_cluster_u32(peer_abort, 1u);
            return false;
        }
    }
}

// Persistent kernel: pair q (q = blockIdx.x / 2) works through its segments
// (its data-parallel tiles, then its stream-K range) of the P = gridDim.x / 2
// pairs' schedule.
template <int MODE>
__global__ void __launch_bounds__(PairCfg::THREADS, 1)
    k_gemm_pair(const __grid_constant__ GemmMaps tm, const TcParams p) {
    using C = PairCfg;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t *full = bar;                       // this CTA's TMA bytes landed
    uint64_t *ready = bar + C::STAGES;          // even CTA: both halves decoded (8 warp arrivals)
    uint64_t *empty = bar + 2 * C::STAGES;      // stage consumed by the MMAs (commit from the even CTA)
    uint64_t *tfull = bar + 3 * C::STAGES;      // accumulators complete (commit from the even CTA)
    uint64_t *tempty = bar + 3 * C::STAGES + 1; // even CTA: accumulators drained (8 warp arrivals)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar + 3 * C::STAGES + 2);
    uint64_t *mdrain = bar + 3 * C::STAGES + 3; // even CTA: every MMA issued has completed
    uint64_t *fixbar = bar + 16;                // NFIX per epilogue warp: partial pieces fetched for finishing
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    auto wtile = [&](int s) { return smem + s * C::STAGE_BYTES; };
    auto atile = [&](int s, int h) { return smem + s * C::STAGE_BYTES + C::W_BYTES + h * C::A_BYTES; };
    auto ctile = [&](int s) { return smem + s * C::STAGE_BYTES + C::W_BYTES + 2 * C::A_BYTES; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = pair_rank();
    const uint32_t peer = rank ^ 1u;
    const uint32_t peer_abort = mapa_u32(smem_u32((const void *)abort_flag), peer);
    const PairPlan pl = make_plan(p, gridDim.x >> 1);
    const int64_t pair_id = blockIdx.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&ready[s], 2 * C::GROUP_WARPS);
            mbar_init(&empty[s], 1);
        }
        mbar_init(tfull, 1);
        mbar_init(tempty, 2 * C::EPI_WARPS);
        mbar_init(mdrain, 1);
        for (int i = 0; i < C::NFIX * C::EPI_WARPS; ++i) mbar_init(&fixbar[i], 1);
        *abort_flag = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc2(tmem_slot, C::TMEM_COLS);
        tmem_relinquish2();
    }
    if (warp == 0 && lane == 0) {
        const int nw = p.ncg > p.nkg ? p.ncg : p.nkg;
        for (int g = 0; g < p.nkg; ++g) prefetch_tmap(&tm.act[g]);
        for (int g = 0; g < nw; ++g) prefetch_tmap(&tm.codes[g]);
        prefetch_tmap(&tm.lact);
        for (int g = 0; g < p.ncg; ++g) {
            prefetch_tmap(&tm.lw[g]);
            if (p.pj[g].out_v4) prefetch_tmap(&tm.out[g]);
        }
        // the first steps' activation and code tiles into L2 while the
        // preceding kernel finishes (L2 stays coherent with its writes)
        SegWalk sw = seg_walk(pl, pair_id);
        PairSeg w;
        if (seg_next(p, pl, sw, w)) {
            const int64_t rowA0 = w.m0 + (int64_t)rank * C::SUB;
            const int64_t ch = w.c0 + (int64_t)rank * C::HN;
            for (int64_t it = 0; it < w.nmain && it < C::STAGES; ++it) {
                const int64_t kk = w.kbeg + it;
                const int kg = MODE == kFwd ? 0 : kgroup_of(p, kk);
                const int32_t k = (int32_t)((kk - p.kg_first[kg]) * C::BK);
                tma_prefetch_2d(&tm.act[kg], k, (int32_t)rowA0);
                if (w.two) tma_prefetch_2d(&tm.act[kg], k, (int32_t)(rowA0 + 256));
                if (MODE == kFwd)
                    tma_prefetch_2d(&tm.codes[w.cg], k / 2, (int32_t)ch);
                else
                    tma_prefetch_2d(&tm.codes[kg], (int32_t)(ch / 2), k);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    pair_sync();  // barriers of both CTAs initialised before any remote arrive
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();     // inputs written by the preceding kernel are visible from here on
    pdl_trigger();

    if (warp == 0) {
        // ------------------------------------------------ TMA producer ----
        if (lane == 0) {
            int64_t g = 0;
            bool alive = true;
            SegWalk sw = seg_walk(pl, pair_id);
            PairSeg w;
            while (alive && seg_next(p, pl, sw, w)) {
                const int64_t rowA0 = w.m0 + (int64_t)rank * C::SUB, rowA1 = rowA0 + 256;
                const int64_t ch = w.c0 + (int64_t)rank * C::HN;
                const uint32_t abytes = (w.two ? 2 : 1) * C::A_BYTES;
                for (int64_t it = 0; it < w.nk; ++it, ++g) {
                    const int s = (int)(g % C::STAGES);
                    const uint32_t ph = (uint32_t)(g / C::STAGES);
                    if (ph > 0 && !pair_wait(&empty[s], (ph - 1) & 1, p.wait_ns, (p.kernel_id << 16) | 1, abort_flag,
                                             peer_abort)) {
                        alive = false;
                        break;
                    }
                    QLORA_STAMP(0, 0, g);
                    if (it < w.nmain) {
                        mbar_arrive_expect_tx(&full[s], abytes + C::C_BYTES);
                        const int64_t kk = w.kbeg + it;
                        const int kg = MODE == kFwd ? 0 : kgroup_of(p, kk);
                        const int32_t k = (int32_t)((kk - p.kg_first[kg]) * C::BK);
                        tma_load_2d(atile(s, 0), &tm.act[kg], &full[s], k, (int32_t)rowA0);
                        if (w.two) tma_load_2d(atile(s, 1), &tm.act[kg], &full[s], k, (int32_t)rowA1);
                        if (MODE == kFwd)
                            tma_load_2d(ctile(s), &tm.codes[w.cg], &full[s], k / 2, (int32_t)ch);
                        else
                            tma_load_2d(ctile(s), &tm.codes[kg], &full[s], (int32_t)(ch / 2), k);
                    } else {
                        const int32_t j = (int32_t)(w.lbeg + it - w.nmain) * C::BK;
                        const int32_t jl = p.pj[w.cg].lcol + j;  // column of the LoRA activations
                        mbar_arrive_expect_tx(&full[s], abytes + C::W_BYTES);
                        tma_load_2d(atile(s, 0), &tm.lact, &full[s], jl, (int32_t)rowA0);
                        if (w.two) tma_load_2d(atile(s, 1), &tm.lact, &full[s], jl, (int32_t)rowA1);
                        if (MODE == kFwd) {
                            tma_load_2d(wtile(s), &tm.lw[w.cg], &full[s], j, (int32_t)ch);
                        } else {
#pragma unroll
                            for (int b = 0; b < 2; ++b)
                                tma_load_2d(wtile(s) + b * 8192, &tm.lw[0], &full[s], (int32_t)(ch + 64 * b), j);
                        }
                    }
                }
            }
            // drain: the last load issued into each stage must have landed
            for (int s = 0; s < C::STAGES; ++s) {
                if (g <= s) break;
                const int64_t last = g - 1 - ((g - 1 - s) % C::STAGES);
                drain_wait(&full[s], (uint32_t)(last / C::STAGES) & 1);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------- MMA issuer (even CTA) ----
        if (rank == 0 && lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(2 * C::SUB, C::BN, 0, MODE == kDx ? 1 : 0);
            int64_t g = 0, tl = 0;
            bool alive = true;
            SegWalk sw = seg_walk(pl, pair_id);
            PairSeg w;
            for (; alive && seg_next(p, pl, sw, w); ++tl) {
                if (tl > 0 && !pair_wait(tempty, (uint32_t)(tl - 1) & 1, p.wait_ns, (p.kernel_id << 16) | 6,
                                         abort_flag, peer_abort))
                    break;
                tc_fence_after();
                for (int64_t it = 0; it < w.nk; ++it, ++g) {
                    const int s = (int)(g % C::STAGES);
                    const uint32_t par = (uint32_t)(g / C::STAGES) & 1;
                    if (!pair_wait(&ready[s], par, p.wait_ns, (p.kernel_id << 16) | 4, abort_flag, peer_abort)) {
                        alive = false;
                        break;
                    }
                    tc_fence_after();
                    QLORA_STAMP(3, 0, g);
                    int nmma = 4;
                    if (it >= w.nmain) {
                        const int rem = p.r - (int)(w.lbeg + it - w.nmain) * C::BK;
                        nmma = rem >= C::BK ? 4 : (rem + 15) / 16;
                    }
                    const uint32_t a0 = smem_u32(atile(s, 0)), a1 = smem_u32(atile(s, 1)), w0 = smem_u32(wtile(s));
                    for (int kk = 0; kk < nmma; ++kk) {
                        const uint64_t bd = MODE == kFwd ? smem_desc_sw128(w0 + kk * 32, 16, 1024)
                                                         : smem_desc_sw128(w0 + kk * 2048, 8192, 1024);
                        const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
                        tc_mma2_bf16(tmem, smem_desc_sw128(a0 + kk * 32, 16, 1024), bd, idesc, acc);
                        if (w.two) tc_mma2_bf16(tmem + 256, smem_desc_sw128(a1 + kk * 32, 16, 1024), bd, idesc, acc);
                    }
                    tc_commit2_both(&empty[s]);
                    QLORA_STAMP(4, 0, g);
                }
                tc_commit2_both(tfull);
            }
            // every MMA issued (also after an abort, when the epilogue may not
            // have waited for the last ones) completes before the pair gives
            // up its operand tiles and TMEM
            if (g > 0) {
                tc_commit2_self(mdrain);
                drain_wait(mdrain, 0);
            }
        }
    } else if (warp < 2 + C::GROUP_WARPS * C::DEC_GROUPS) {
        // ------------------------------ decode groups (alternate k-steps) ----
        const int dw = warp - 2;
        const int grp = dw / C::GROUP_WARPS;
        const int dt = (dw % C::GROUP_WARPS) * 32 + lane;  // 0..127 within the group
        const int64_t kblocks = p.w_cols / kBlock;
        const uint32_t ready_addr0 = mapa_u32(smem_u32(ready), 0);
        uint32_t dst[8], csrc[2];
        int b2 = 0, nl = 0;
        if (MODE == kFwd) {
            // row dt of the K-major, 128-byte swizzled W' half-tile
#pragma unroll
            for (int c = 0; c < 8; ++c) dst[c] = (uint32_t)((dt >> 3) * 1024 + (dt & 7) * 128 + ((c ^ (dt & 7)) << 4));
            // 32-byte code rows, 32-byte swizzle: half h sits at h ^ bit 2 of the row
#pragma unroll
            for (int h = 0; h < 2; ++h) csrc[h] = (uint32_t)(dt * 32 + ((h ^ ((dt >> 2) & 1)) << 4));
        } else {
            // W row it*64 + nl (a K-group row of the MN-major operand), column block b2
            const int nlo = dt & 7, nhi = dt >> 4;
            b2 = (dt >> 3) & 1;
            nl = nhi * 8 + nlo;
#pragma unroll
            for (int c = 0; c < 8; ++c) dst[c] = (uint32_t)(b2 * 8192 + nhi * 1024 + nlo * 128 + ((c ^ nlo) << 4));
            // 64-byte code rows, 64-byte swizzle: 16-byte chunk q sits at q ^ ((row >> 1) & 3)
#pragma unroll
            for (int h = 0; h < 2; ++h) csrc[h] = (uint32_t)(nl * 64 + (((b2 * 2 + h) ^ ((nl >> 1) & 3)) << 4));
        }
        // This group's steps (global step g with g % DEC_GROUPS == grp) are
        // walked with a cursor; the absmax code and group scale of the next
        // step are loaded before the current step is waited for and decoded.
        // (only what the decode needs of a segment: its first step and
        // main steps, its column tile and its length)
        struct Cursor {
            SegWalk sw;
            bool live;
            int cg;
            int64_t it, g, nk, nmain, kbeg, c0;
        };
        auto enter = [&](Cursor &c) {
            PairSeg w = {};
            c.live = seg_next(p, pl, c.sw, w);
            c.it = 0;
            c.nk = w.nk;
            c.nmain = w.nmain;
            c.kbeg = w.kbeg;
            c.c0 = w.c0;
            c.cg = w.cg;
        };
        auto advance = [&](Cursor &c) {
            ++c.it;
            ++c.g;
            if (c.live && c.it >= c.nk) enter(c);
        };
        // The block's reconstructed absmax is a' = fp32(qv) * sv + mv: the
        // double-quantized code, its group scale and the weight's mean, or
        // (0, 0, a) for an fp32 absmax a (0 * 0 + a is exactly a).
        auto fetch = [&](const Cursor &c, int &qv, float &sv, float &mv) {
            qv = 0;
            sv = 0.0f;
            mv = 0.0f;
            if (!c.live || c.it >= c.nmain) return false;
            const int64_t ch = c.c0 + (int64_t)rank * C::HN;
            const int64_t kk = c.kbeg + c.it;
            const int kg = MODE == kFwd ? 0 : kgroup_of(p, kk);
            const TcProj &pw = p.pj[MODE == kFwd ? c.cg : kg];
            const int64_t wrow = MODE == kFwd ? ch + dt : (kk - p.kg_first[kg]) * C::BK + nl;
            const int64_t kb = MODE == kFwd ? kk : ch / kBlock + b2;
            if (wrow >= pw.rows || kb >= kblocks) return false;
            const int64_t bidx = wrow * kblocks + kb;
            if (pw.absmax) {
                mv = __ldg(pw.absmax + bidx);
            } else {
                qv = __ldg(pw.q + bidx);
                sv = __ldg(pw.s2 + (bidx >> 8));
                mv = __ldg(pw.mean);
            }
            return true;
        };
        Cursor cur;
        cur.sw = seg_walk(pl, pair_id);
        cur.g = 0;
        enter(cur);
        for (int i = 0; i < grp; ++i) advance(cur);
        Cursor nxt = cur;
        for (int i = 0; i < C::DEC_GROUPS; ++i) advance(nxt);
        int qv, qn;
        float sv, sn, mv, mn;
        bool valid = fetch(cur, qv, sv, mv);
        while (cur.live) {
            const bool valid_n = fetch(nxt, qn, sn, mn);
            const int s = (int)(cur.g % C::STAGES);
            const uint32_t par = (uint32_t)(cur.g / C::STAGES) & 1;
            if (!pair_wait(&full[s], par, p.wait_ns, (p.kernel_id << 16) | 2, abort_flag, peer_abort)) break;
            if (lane == 0 && dw % C::GROUP_WARPS == 0) QLORA_STAMP(1, 0, cur.g);
            if (cur.it < cur.nmain) {
                uint8_t *wt = wtile(s);
                const uint8_t *ct = ctile(s);
                uint32_t o[8][4];
                if (valid) {
                    const Nf4Table tab = make_table(dq_absmax((int8_t)qv, sv, mv), p.tab);
                    uint4 cw[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) cw[h] = *reinterpret_cast<const uint4 *>(ct + csrc[h]);
                    const uint32_t wv[8] = {cw[0].x, cw[0].y, cw[0].z, cw[0].w, cw[1].x, cw[1].y, cw[1].z, cw[1].w};
#pragma unroll
                    for (int c = 0; c < 8; ++c) decode8(tab, wv[c], o[c]);
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
            if (lane == 0 && dw % C::GROUP_WARPS == 0) {
                QLORA_STAMP(2, 0, cur.g);
                QLORA_STAMP(7, 1, cur.g);
            }
            if (lane == 0) mbar_arrive_cluster(ready_addr0 + (uint32_t)(s * 8));
            cur = nxt;
            qv = qn;
            sv = sn;
            mv = mn;
            valid = valid_n;
            for (int i = 0; i < C::DEC_GROUPS; ++i) advance(nxt);
        }
    } else {
        // --------------------------------------------------- epilogue ----
        // Epilogue warp e (one per TMEM lane quarter, quarter = warp % 4)
        // reads lanes 32 * quarter .. + 31 (one row of each 128-row sub-tile
        // per thread), 64 accumulator columns per wait (batch b = 4 * sub +
        // column block). The accumulators are released to the next segment's
        // MMAs right after the last read. Output rows go through the warp's
        // 4 KB staging buffer (32 rows x 128 bytes, 16-byte chunks rotated by
        // row so neither side conflicts on banks) and leave as whole 128-byte
        // lines, four rows per store instruction.
        //
        // A partial tile goes to the pair's slot in this warp's own order:
        // [CTA][warp][batch][8-column chunk][lane][8 fp32], so every store
        // instruction writes 1 KB of consecutive bytes. Finishing a tile in
        // the pair's last segment, the warp fetches the matching 8 KB pieces
        // of the other contributors' slots into the (now idle) stage buffers
        // with bulk copies, NFIX in flight; finishing one earlier, it loads
        // them from global memory. It adds them in pair order.
        const int ew = warp - (2 + C::GROUP_WARPS * C::DEC_GROUPS);  // 0..3
        const int quarter = warp & 3;
        uint8_t *stg = smem + C::EPI_OFF + ew * 4096;
        const uint32_t tempty_addr0 = mapa_u32(smem_u32(tempty), 0);
        uint8_t *fixbuf = smem + ew * (C::NFIX * 8192);  // NFIX 8 KB buffers of this warp
        // pieces fetched / consumed, counted over the whole launch: a pair may
        // finish two shared tiles, and the piece ring's barriers keep their
        // phases from one to the next
        int fx_issued = 0, fx_waited = 0;
        int64_t tl = 0;
        SegWalk sw = seg_walk(pl, pair_id);
        PairSeg w;
        for (; seg_next(p, pl, sw, w); ++tl) {
            if (!pair_wait(tfull, (uint32_t)tl & 1, p.wait_ns, (p.kernel_id << 16) | 5, abort_flag, peer_abort))
                break;
            if (ew == 0 && lane == 0) QLORA_STAMP(5, 0, tl);
            tc_fence_after();
            const int nb = w.two ? C::NBATCH : C::NBATCH / 2;
            // a shared tile: contributors h .. h + n - 1, this pair is number m
            int64_t h = pair_id;
            int n = 1;
            if (w.role != kSegFull) {
                if (w.role == kSegPart) h = head_pair(pl, pair_id, w.t);
                n = (int)(head_contrib_end(pl, h, w.t) - h);
            }
            const int m = (int)(pair_id - h);
            bool finish = true;
            if (n > 1) {
                uint32_t old = 0;
                if (lane == 0)
                    old = atom_add_acq_rel_gpu(p.flags + kSkReadyWords + (h * 2 + rank) * C::EPI_WARPS + ew, 1u);
                finish = __shfl_sync(0xffffffffu, old, 0) == (uint32_t)(n - 1);
            }
            // the others' partials this warp adds when it finishes the tile:
            // piece i = (batch b, other contributor qi), the one of pair
            // h + j with j = qi (before this pair) or qi + 1 (after it); the
            // head's partial is in its head slot, the others' in their tail slots
            const int nq = finish ? n - 1 : 0;
            if (nq > C::NFIX) {
                // (the schedule never shares a tile this widely)
                if (lane == 0) {
                    record_error((p.kernel_id << 16) | 9);
                    *abort_flag = 1;
                    st_cluster_u32(peer_abort, 1u);
                }
                break;
            }
            // The pieces go through the stage ring (bulk copies, NFIX in
            // flight) only when this is the pair's last segment: the ring is
            // idle then (every load issued has been consumed by the MMAs).
            // A pair finishing a tile with more segments to come (a tail that
            // arrived last) reads the partials from global memory instead.
            SegWalk nx = sw;
            PairSeg wn;
            const bool use_ring = !seg_next(p, pl, nx, wn);
            const int nitems = use_ring ? nq * nb : 0;
            const int fx0 = fx_issued;  // this segment's piece i is piece fx0 + i of the launch
            auto other = [&](int qi) { return qi < m ? qi : qi + 1; };
            auto slot_of = [&](int64_t q, int head) { return p.slots + (q * 2 + head) * kSlotFloats; };
            auto ready_of = [&](int64_t q, int head) { return p.flags + ((q * 2 + head) * 2 + rank) * C::EPI_WARPS + ew; };
            auto fetch_piece = [&](int i) {
                if (i >= nitems) return;
                const int gi = fx0 + i;
                fx_issued = gi + 1;
                if (lane != 0) return;
                const int b = i / nq;
                const int j = other(i % nq);
                const float *src = slot_of(h + j, j == 0) + (((int64_t)rank * C::EPI_WARPS + ew) * C::NBATCH + b) * 2048;
                uint64_t *fb = &fixbar[ew * C::NFIX + gi % C::NFIX];
                mbar_arrive_expect_tx(fb, 8192);
                bulk_g2s(fixbuf + (gi % C::NFIX) * 8192, src, 8192, fb);
            };
            if (nq > 0) {
                bool ok = true;
                if (lane == 0) {
                    for (int qi = 0; qi < nq && ok; ++qi) {
                        const int j = other(qi);
                        ok = flag_wait(ready_of(h + j, j == 0), p.wait_ns, (p.kernel_id << 16) | 7, abort_flag,
                                       peer_abort);
                    }
                    if (ok) asm volatile("fence.proxy.async.global;" ::: "memory");
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok) break;
                for (int i = 0; i < C::NFIX; ++i) fetch_piece(i);
            }
            bool alive = true;
            for (int sub = 0; sub < 2 && alive; ++sub) {
                if (sub == 1 && !w.two) break;
                const int64_t rbase = w.m0 + sub * 256 + (int64_t)rank * C::SUB + quarter * 32;  // warp's first row
                const int64_t row = rbase + lane;
#pragma unroll 1
                for (int cb = 0; cb < 4; ++cb) {
                    const int col = cb * 64;
                    const int b = sub * 4 + cb;
                    uint32_t v[64];
                    const uint32_t ta = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(sub * 256 + col);
                    tmem_ld_32x32b_x32(ta, *reinterpret_cast<uint32_t(*)[32]>(v));
                    tmem_ld_32x32b_x32(ta + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
                    tmem_ld_wait();
                    if (sub == (w.two ? 1 : 0) && cb == 3) {
                        // every accumulator column this warp owns has been read:
                        // the MMAs of the next segment may overwrite them
                        tc_fence_before();
                        __syncwarp();
                        if (ew == 0 && lane == 0) QLORA_STAMP(6, 0, tl);
                        if (lane == 0) mbar_arrive_cluster(tempty_addr0);
                    }
                    if (!finish) {
                        float *dst = slot_of(pair_id, m == 0) +
                                     (((int64_t)rank * C::EPI_WARPS + ew) * C::NBATCH + b) * 2048;
#pragma unroll
                        for (int jc = 0; jc < 8; ++jc) {
                            uint32_t pk[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) pk[e] = v[8 * jc + e];
                            st_global_v8(dst + (jc * 32 + lane) * 8, pk);
                        }
                        continue;
                    }
                    if (nq > 0) {
                        // this batch's pieces (nq <= NFIX: all in the ring at once)
                        for (int qi = 0; qi < nq && alive && use_ring; ++qi) {
                            const int gi = fx0 + b * nq + qi;
                            alive = pair_wait(&fixbar[ew * C::NFIX + gi % C::NFIX], (uint32_t)(gi / C::NFIX) & 1,
                                              p.wait_ns, (p.kernel_id << 16) | 8, abort_flag, peer_abort);
                            if (alive) fx_waited = gi + 1;
                        }
                        if (!alive) break;
                        // Pair order, ((P_0 + P_1) + ...) + P_{n-1}, with this
                        // pair's accumulators (v) as P_m: the terms before P_m
                        // are first folded, in order, into one buffer Q (P_0's
                        // piece in the ring, else this pair's own tail slot,
                        // unused while it finishes this tile); then v = v + Q,
                        // the same as Q + v, and v += P_{m+1}, ... in order.
                        auto piece = [&](int j) -> float * {
                            if (use_ring)
                                return reinterpret_cast<float *>(
                                    fixbuf + ((fx0 + b * nq + (j < m ? j : j - 1)) % C::NFIX) * 8192);
                            return slot_of(h + j, j == 0) + (((int64_t)rank * C::EPI_WARPS + ew) * C::NBATCH + b) * 2048;
                        };
                        float *q = nullptr;
                        if (m >= 2) {
                            q = use_ring ? piece(0)
                                         : slot_of(pair_id, 0) + (((int64_t)rank * C::EPI_WARPS + ew) * C::NBATCH + b) * 2048;
#pragma unroll 1
                            for (int j = use_ring ? 1 : 0; j < m; ++j) {
                                const float *src = piece(j);
#pragma unroll
                                for (int jc = 0; jc < 8; ++jc) {
                                    const int o = (jc * 32 + lane) * 8;
                                    float4 x0 = ld_f4_gpu(src + o), x1 = ld_f4_gpu(src + o + 4);
                                    if (j > 0) {
                                        const float4 y0 = ld_f4_gpu(q + o), y1 = ld_f4_gpu(q + o + 4);
                                        x0 = make_float4(y0.x + x0.x, y0.y + x0.y, y0.z + x0.z, y0.w + x0.w);
                                        x1 = make_float4(y1.x + x1.x, y1.y + x1.y, y1.z + x1.z, y1.w + x1.w);
                                    }
                                    *reinterpret_cast<float4 *>(q + o) = x0;
                                    *reinterpret_cast<float4 *>(q + o + 4) = x1;
                                }
                            }
                        }
#pragma unroll 1
                        for (int j = 0; j < n; ++j) {
                            if (j == m || (j > 0 && j < m)) continue;
                            const float *src = j == 0 && m >= 2 ? q : piece(j);
#pragma unroll
                            for (int jc = 0; jc < 8; ++jc) {
                                const float4 a0 = ld_f4_gpu(src + (jc * 32 + lane) * 8);
                                const float4 a1 = ld_f4_gpu(src + (jc * 32 + lane) * 8 + 4);
                                const float add[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                                for (int e = 0; e < 8; ++e)
                                    v[8 * jc + e] = __float_as_uint(__uint_as_float(v[8 * jc + e]) + add[e]);
                            }
                        }
                        __syncwarp();  // every lane has read the buffers before they are refilled
                        for (int qi = 0; qi < nq; ++qi) fetch_piece(b * nq + qi + C::NFIX);
                    }
                    const TcProj &po = p.pj[w.cg];
                    const int64_t ncol = po.ncols - (w.c0 + col);  // valid columns from here
                    if (po.out_v4) {
                        // the previous batch's store has read the staging tile
                        if (lane == 0) bulk_wait_read<0>();
                        __syncwarp();
                        // row `lane` into the staging tile: chunk c (8 columns)
                        // at c ^ (lane & 7), the tensor map's 128-byte swizzle
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            uint4 pk;
                            pk.x = pack_bf16x2(__uint_as_float(v[8 * c + 0]), __uint_as_float(v[8 * c + 1]));
                            pk.y = pack_bf16x2(__uint_as_float(v[8 * c + 2]), __uint_as_float(v[8 * c + 3]));
                            pk.z = pack_bf16x2(__uint_as_float(v[8 * c + 4]), __uint_as_float(v[8 * c + 5]));
                            pk.w = pack_bf16x2(__uint_as_float(v[8 * c + 6]), __uint_as_float(v[8 * c + 7]));
                            *reinterpret_cast<uint4 *>(stg + lane * 128 + ((c ^ (lane & 7)) << 4)) = pk;
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        // one TMA store of the 32 x 64 box; rows and columns
                        // past the output's edge are clipped by the unit
                        if (lane == 0 && rbase < p.M) {
                            tma_store_2d(&tm.out[w.cg], stg, (int32_t)(w.c0 + col), (int32_t)rbase);
                            bulk_commit();
                        }
                        continue;
                    }
                    if (row >= p.M) continue;
                    uint16_t *dstp = po.out + row * po.ldo + w.c0 + col;
#pragma unroll
                    for (int e = 0; e < 64; ++e)
                        if (e < ncol) dstp[e] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[e])));
                }
            }
            if (!alive) break;
            if (!finish) {
                // this warp's share of the partial tile is written: raise its flag
                __syncwarp();
                if (lane == 0) {
                    __threadfence();
                    st_release_gpu(ready_of(pair_id, m == 0), 1u);
                }
            }
        }
        // the output stores complete before the CTA leaves
        if (lane == 0) bulk_wait_all();
        // after an abort: let the fetches still in flight land before the
        // shared memory is given up
        if (lane == 0) {
            for (int i = fx_waited; i < fx_issued; ++i)
                drain_wait(&fixbar[ew * C::NFIX + i % C::NFIX], (uint32_t)(i / C::NFIX) & 1);
        }
    }
    tc_fence_before();
    __syncwarp();
    pair_sync();  // both CTAs done with the MMAs' shared memory and TMEM
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc2(tmem, C::TMEM_COLS);
    }
}

}  // namespace qlora
