// stream_probe.cu -- diagnostic program (not part of the library): how fast
// can one launch read a packed weight of the gate projection's size
// (14336 rows x 2048 bytes = 29.4 MB) from HBM into shared memory, with no
// work on the data? The reading pattern is the few-token forward's: tasks of
// 32 rows x 128 bytes (one TMA box), split evenly over 148 CTAs x 16 warps,
// every warp keeping two tasks in flight. Reported: the single-launch time,
// the time per launch back to back (six weight copies, more than L2 holds),
// and both for an empty launch of the same shape (no warp has a task).
//
//   nvcc -gencode arch=compute_103a,code=sm_103a -O3 -o stream_probe \
//        bit_quantized_lora_double_b300/stream_probe.cu -lcuda && ./stream_probe
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <vector>

namespace {

constexpr int kWarps = 16, kSlots = 2, kTaskBytes = 4096, kRows = 32;

__device__ __forceinline__ uint32_t su(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ bool bar_try(uint64_t *b, uint32_t ph) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(su(b)), "r"(ph)
        : "memory");
    return ok != 0;
}

// Every wait is bounded: on running out the warp records an error, waits
// (again bounded) for its own loads in flight and returns.
__global__ void __launch_bounds__(kWarps * 32, 1)
    k_stream(const __grid_constant__ CUtensorMap tm, int tasks_per_row, int T, int W, int *err) {
    extern __shared__ __align__(1024) uint8_t sm[];
    uint8_t *base = (uint8_t *)(((uintptr_t)sm + 1023) & ~(uintptr_t)1023);
    __shared__ uint64_t bars[kWarps * kSlots];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gw = blockIdx.x * kWarps + warp;
    if (gw >= W) return;
    const int t0 = (int)((long long)gw * T / W), t1 = (int)((long long)(gw + 1) * T / W), n = t1 - t0;
    uint64_t *f = bars + kSlots * warp;
    if (lane == 0) {
        for (int s = 0; s < kSlots; ++s)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su(&f[s])) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    auto issue = [&](int s, int x) {
        const int rt = x / tasks_per_row, kc = x - rt * tasks_per_row;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su(&f[s])), "r"(kTaskBytes)
                     : "memory");
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
            "[%2];" ::"r"(su(base + (warp * kSlots + s) * kTaskBytes)),
            "l"((uint64_t)&tm), "r"(su(&f[s])), "r"(kc * 128), "r"(rt * kRows)
            : "memory");
    };
    if (lane == 0)
        for (int s = 0; s < kSlots && s < n; ++s) issue(s, t0 + s);
    for (int i = 0; i < n; ++i) {
        const int s = i % kSlots;
        const uint32_t ph = (i / kSlots) & 1;
        long long it = 0;
        while (!bar_try(&f[s], ph)) {
            if (++it > (1ll << 26)) {
                if (lane == 0) atomicExch(err, 1);
                for (int q = i; q < i + kSlots && q < n; ++q)
                    for (long long j = 0; j < (1ll << 26) && !bar_try(&f[q % kSlots], (q / kSlots) & 1); ++j) {
                    }
                return;
            }
        }
        __syncwarp();
        if (lane == 0 && i + kSlots < n) issue(s, t0 + i + kSlots);
    }
}

typedef CUresult (*EncodeTiled)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

}  // namespace

int main() {
    const int N = 14336, KB = 2048, copies = 6, tasks_per_row = KB / 128;
    const size_t bytes = (size_t)N * KB;
    const int T = (N / kRows) * tasks_per_row, W = std::min(T, 148 * kWarps), grid = (W + kWarps - 1) / kWarps;
    const int smem = kWarps * kSlots * kTaskBytes + 1024;
    std::vector<uint8_t *> d(copies);
    for (auto &p : d) {
        if (cudaMalloc(&p, bytes) != cudaSuccess) return 1;
        cudaMemset(p, 1, bytes);
    }
    int *err;
    cudaMalloc(&err, 4);
    cudaMemset(err, 0, 4);
    EncodeTiled enc = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", (void **)&enc, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        !enc)
        return 1;
    std::vector<CUtensorMap> tm(copies);
    for (int c = 0; c < copies; ++c) {
        const cuuint64_t dims[2] = {(cuuint64_t)KB, (cuuint64_t)N}, strides[1] = {(cuuint64_t)KB};
        const cuuint32_t box[2] = {128, kRows}, es[2] = {1, 1};
        if (enc(&tm[c], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, d[c], dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE))
            return 1;
    }
    cudaFuncSetAttribute(k_stream, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    // best of several timings of `reps` launches between two events, per launch
    auto time = [&](int reps, int w) {
        float best = 1e9f;
        for (int it = 0; it < 12; ++it) {
            cudaEventRecord(e0);
            for (int k = 0; k < reps; ++k)
                k_stream<<<grid, kWarps * 32, smem>>>(tm[(it * reps + k) % copies], tasks_per_row, T, w, err);
            cudaEventRecord(e1);
            cudaEventSynchronize(e1);
            float ms;
            cudaEventElapsedTime(&ms, e0, e1);
            if (it >= 2) best = std::min(best, ms / reps);
        }
        return best * 1e3f;
    };
    const float single = time(1, W), b2b = time(copies, W), e_single = time(1, 0), e_b2b = time(copies, 0);
    int h = 0;
    cudaMemcpy(&h, err, 4, cudaMemcpyDeviceToHost);
    printf("{\"bytes\": %zu, \"single_us\": %.2f, \"back_to_back_us\": %.2f, \"empty_single_us\": %.2f, "
           "\"empty_back_to_back_us\": %.2f, \"single_gbs\": %.0f, \"back_to_back_gbs\": %.0f, \"error\": %d, "
           "\"cuda\": \"%s\"}\n",
           bytes, single, b2b, e_single, e_b2b, bytes / (single * 1e-6) / 1e9, bytes / (b2b * 1e-6) / 1e9, h,
           cudaGetErrorString(cudaGetLastError()));
    return h != 0;
}
