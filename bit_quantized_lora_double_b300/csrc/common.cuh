// common.cuh -- device helpers shared by the kernels of the QLoRA library.
//
// Contents: format constants, the device error word used by bounded waits,
// PTX wrappers (mbarrier, TMA, tcgen05, proxy fences) for sm_103a, and the
// register-only NF4 decoder (code nibbles -> bf16 pairs through a per-block
// scaled 16-entry table held as byte planes and selected with PRMT).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "nf4_table.h"

namespace qlora {

constexpr int kBlock = 64;    // weights per NF4 block (one absmax each)
constexpr int kGroup = 256;   // blocks per second-level (fp32 scale) group

// Level tables: [0] NF4, [1] the INT4 baseline; the encode thresholds with
// them. Kernels take the table id as a launch-uniform argument.
enum { kTableNF4 = 0, kTableINT4 = 1 };
__constant__ float c_levels_q4[2][16] = {QLORA_NF4_LEVELS, QLORA_INT4_LEVELS};
__constant__ float c_thresholds_q4[2][15] = {QLORA_NF4_THRESHOLDS, QLORA_INT4_THRESHOLDS};

// ---------------------------------------------------------------------------
// Device error word: the first bounded wait that runs out records
// (kernel id << 16 | wait site) here; the host reads and clears it.
// ---------------------------------------------------------------------------
__device__ unsigned int g_error_word = 0;

__device__ __forceinline__ void record_error(unsigned int code) {
    atomicCAS(&g_error_word, 0u, code);
}

// ---------------------------------------------------------------------------
// Small PTX wrappers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait that lets the hardware suspend the thread until the phase
// completes or about `hint_ns` nanoseconds pass, so that waiting warps do not
// take issue slots from working ones.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
constexpr uint32_t kWaitHintNs = 20000;

// 2-D TMA tile load into shared memory, completion counted on `bar` (bytes).
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar, int32_t x,
                                            int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
        "[%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}

// TMA tile store (shared -> global) of one 2-D box, tracked as a bulk group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *src, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(src)), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N committed bulk groups of this thread still read
// shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Bring one 2-D box of a tensor into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- tcgen05 (5th-generation tensor core, accumulators in TMEM) ----------
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread
// has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns from TMEM into registers.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor for tcgen05 (sm_100 family format):
// start address, leading/stride byte offsets (all >> 4), version 1, and the
// swizzle mode (2 = 128-byte swizzle). Tiles are 1024-byte aligned, so the
// base offset field stays 0.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;  // SWIZZLE_128B
    return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, dense.
// a_mn / b_mn: operand is MN-major (1) or K-major (0).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
    return (1u << 4)                          // D format: f32
           | (1u << 7)                        // A format: bf16
           | (1u << 10)                       // B format: bf16
           | ((uint32_t)a_mn << 15)           // A major
           | ((uint32_t)b_mn << 16)           // B major
           | ((uint32_t)(N >> 3) << 17)       // N / 8
           | ((uint32_t)(M >> 4) << 24);      // M / 16
}

// ---------------------------------------------------------------------------
// NF4 decode through a per-block scaled table.
//
// For one block (fixed row n, 64 consecutive k) with reconstructed absmax a',
// entry i of the table is bf16_rne(fp32(L[i] * a')): exactly the dequantized
// value of code i, so the table lookup is bit-identical to decoding element
// by element. The 16 entries live in 8 registers as byte planes: lo[q] holds
// the low bytes of entries 4q..4q+3 and hi[q] their high bytes, so PRMT can
// select four entries at a time.
// ---------------------------------------------------------------------------
struct Nf4Table {
    uint32_t lo[4], hi[4];
};

__device__ __forceinline__ float dq_absmax(int8_t q, float s2, float mean) {
    return __fadd_rn(__fmul_rn(static_cast<float>(q), s2), mean);
}

__device__ __forceinline__ Nf4Table make_table(float a, int tab = kTableNF4) {
    const float *L = c_levels_q4[tab];
    uint32_t p[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        __nv_bfloat162 v = __floats2bfloat162_rn(__fmul_rn(L[2 * j], a), __fmul_rn(L[2 * j + 1], a));
        p[j] = *reinterpret_cast<uint32_t *>(&v);  // entry 2j in the low half
    }
    Nf4Table t;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        t.lo[q] = prmt(p[2 * q], p[2 * q + 1], 0x6420);
        t.hi[q] = prmt(p[2 * q], p[2 * q + 1], 0x7531);
    }
    return t;
}

// Decodes 8 packed codes w (byte j = code(2j) << 4 | code(2j+1)) into four
// bf16 pairs o[j] = (elem 2j in the low half, elem 2j+1 in the high half).
__device__ __forceinline__ void decode8(const Nf4Table &t, uint32_t w, uint32_t (&o)[4]) {
    const uint32_t s = w & 0x77777777u;  // entry index within a half-table
    const uint32_t z = w << 4;           // msb of byte j = bit 3 of code(2j+1)
    // Byte masks: 0xFF where the code is >= 8 (sign-replicate mode of PRMT).
    // Selector nibbles of the low half-word address codes (1,0,3,2), of the
    // high half-word codes (5,4,7,6).
    const uint32_t mA = prmt(w, z, 0x9D8C);
    const uint32_t mB = prmt(w, z, 0xBFAE);
    const uint32_t sB = s >> 16;
    uint32_t loA = (prmt(t.lo[2], t.lo[3], s) & mA) | (prmt(t.lo[0], t.lo[1], s) & ~mA);
    uint32_t hiA = (prmt(t.hi[2], t.hi[3], s) & mA) | (prmt(t.hi[0], t.hi[1], s) & ~mA);
    uint32_t loB = (prmt(t.lo[2], t.lo[3], sB) & mB) | (prmt(t.lo[0], t.lo[1], sB) & ~mB);
    uint32_t hiB = (prmt(t.hi[2], t.hi[3], sB) & mB) | (prmt(t.hi[0], t.hi[1], sB) & ~mB);
    // byte order in loA/hiA is codes (1,0,3,2): interleave into bf16 pairs
    o[0] = prmt(loA, hiA, 0x4051);
    o[1] = prmt(loA, hiA, 0x6273);
    o[2] = prmt(loB, hiB, 0x4051);
    o[3] = prmt(loB, hiB, 0x6273);
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

}  // namespace qlora
