// qlora_lib.cu -- the C ABI (include/qlora.h): argument validation, workspace
// layout and kernel launches. All kernels are compiled in this one
// translation unit so they share the device error word.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>
#include <algorithm>

#include "qlora.h"

#include "common.cuh"
#include "codec.cuh"
#include "lora_simt.cuh"
#include "gemm_tc.cuh"

using namespace qlora;

namespace {

thread_local std::string t_last_error;
int64_t g_wait_limit = 0;  // 0: default

qlora_status fail(qlora_status st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return st;
}

qlora_status ok() {
    t_last_error.clear();
    return QLORA_OK;
}

inline bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

constexpr int64_t kMaxDim = int64_t(1) << 31;

// ---- optional profiling of our own launches (qlora_profile_start/stop) ----
struct ProfRec {
    cudaEvent_t a, b;
    int kind;
};
std::vector<ProfRec> g_prof;
bool g_prof_on = false;
int g_prof_count[QLORA_KERNEL_KINDS];

struct ProfScope {
    int kind;
    cudaStream_t s;
    cudaEvent_t a = nullptr;
    ProfScope(int k, cudaStream_t st) : kind(k), s(st) {
        if (!g_prof_on) return;
        g_prof_count[k]++;
        if (cudaEventCreate(&a) == cudaSuccess) cudaEventRecord(a, s);
    }
    ~ProfScope() {
        if (!g_prof_on || !a) return;
        cudaEvent_t b;
        if (cudaEventCreate(&b) == cudaSuccess) {
            cudaEventRecord(b, s);
            g_prof.push_back({a, b, kind});
        }
    }
};

qlora_status launch_check(const char *what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(QLORA_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
    return QLORA_OK;
}

bool valid_dims(int64_t rows, int64_t cols) {
    return rows >= 0 && cols > 0 && cols % kBlock == 0 && rows < kMaxDim && cols < kMaxDim;
}

qlora_status check_weight(const qlora_nf4_weight *w, bool need_rows) {
    if (!w) return fail(QLORA_ERR_NULL, "weight descriptor is NULL");
    if (!valid_dims(w->rows, w->cols))
        return fail(QLORA_ERR_SHAPE, "weight shape [%lld, %lld]: need rows >= 0, cols > 0, cols %% 64 == 0",
                    (long long)w->rows, (long long)w->cols);
    if (need_rows && w->rows == 0) return fail(QLORA_ERR_SHAPE, "weight has 0 rows");
    if (!w->codes || !w->absmax_q || !w->absmax_scale || !w->absmax_mean)
        return fail(QLORA_ERR_NULL, "weight descriptor has a NULL array");
    if (!al16(w->codes) || !al16(w->absmax_q) || !al16(w->absmax_scale) || !al16(w->absmax_mean))
        return fail(QLORA_ERR_ALIGN, "weight arrays must be 16-byte aligned");
    return QLORA_OK;
}

// Workspace carving helper: 256-byte aligned slices.
struct Carve {
    char *base;
    size_t off = 0;
    explicit Carve(void *b) : base(static_cast<char *>(b)) {}
    template <class T>
    T *take(size_t count) {
        T *p = reinterpret_cast<T *>(base ? base + off : nullptr);
        off = up(off + count * sizeof(T), 256);
        return p;
    }
};

// ---- quantize workspace: absmax fp32 [nb], group sums fp64 [ng], two
// ping-pong fp64 buffers of ceil(ng / 256) for the upper tree levels.
size_t quantize_ws(int64_t rows, int64_t cols, float **absmax, double **gsum, double **buf0, double **buf1,
                   void *ws) {
    const int64_t nb = rows * cols / kBlock, ng = cdiv(nb, kGroup), nl = cdiv(ng, 256) + 1;
    Carve c(ws);
    float *a = c.take<float>(nb);
    double *g = c.take<double>(ng);
    double *b0 = c.take<double>(nl);
    double *b1 = c.take<double>(nl);
    if (absmax) *absmax = a;
    if (gsum) *gsum = g;
    if (buf0) *buf0 = b0;
    if (buf1) *buf1 = b1;
    return c.off;
}

// ---- linear workspaces
// The LoRA operands of the tensor-core path are zero-padded to rp = 64 *
// ceil(r / 64) columns so every TMA box lies inside its tensor.
inline int lora_pad(int r) { return (int)up((size_t)r, 64); }

// Tokens at or above which the tensor-core path runs.
constexpr int64_t kTcMinM = 64;

// Split of one skinny tcgen05 pass: output rows in 128-row tiles, rank in
// 64-wide column tiles, contraction in chunks of steps_per_chunk x 64.
struct SkPlan {
    int64_t rows, rows_pad, L, spc, chunks;
    int zt;
    size_t part_floats;
};
SkPlan sk_plan(int64_t rows, int64_t L, int rp) {
    SkPlan p;
    p.rows = rows;
    p.rows_pad = (int64_t)up((size_t)rows, 128);
    p.L = L;
    p.zt = rp / 64;
    const int64_t tiles = p.rows_pad / 128 * p.zt;
    const int64_t steps = std::max<int64_t>(1, cdiv(L, 64));
    const int64_t ch = std::min<int64_t>(steps, std::max<int64_t>(1, cdiv(2 * 148, tiles)));
    p.spc = cdiv(steps, ch);
    p.chunks = cdiv(steps, p.spc);
    p.part_floats = (size_t)p.zt * p.chunks * p.rows_pad * 64;
    return p;
}

// Contraction splits of the fused GEMM: split only when the output tiles fill
// less than three quarters of the 148 SMs, keeping >= 4 k-steps per split.
struct GemmSplit {
    int splits;
    int64_t steps_per_split;
};
GemmSplit gemm_split(int64_t M, int64_t Nd, int64_t nk_main) {
    const int64_t tiles = cdiv(Nd, 256) * cdiv(M, 256);
    int64_t sp = 1;
    if (tiles * 4 < 3 * 148) sp = std::max<int64_t>(1, std::min<int64_t>({148 / tiles, nk_main / 4, 8}));
    const int64_t sps = cdiv(nk_main, sp);
    return {(int)cdiv(nk_main, sps), sps};
}

struct FwdWs {
    uint16_t *sU, *Bp, *Ap;
    float *part;
};
size_t fwd_ws(int64_t M, int64_t N, int64_t K, int r, void *ws, FwdWs *out) {
    const int rp = lora_pad(r);
    const bool tc = M >= kTcMinM;
    Carve c(ws);
    uint16_t *sU = c.take<uint16_t>((size_t)M * rp);
    uint16_t *Bp = c.take<uint16_t>(tc ? (size_t)N * rp : 0);
    uint16_t *Ap = c.take<uint16_t>(tc ? (size_t)rp * K : 0);
    size_t pf = 0;
    if (tc) {
        const GemmSplit g = gemm_split(M, N, K / 64);
        pf = std::max(sk_plan(M, K, rp).part_floats, g.splits > 1 ? (size_t)g.splits * M * N : (size_t)0);
    }
    float *part = c.take<float>(pf);
    if (out) *out = FwdWs{sU, Bp, Ap, part};
    return c.off;
}

struct GradSplit {
    int64_t rows_per_chunk, nchunks;
};
GradSplit grad_split(int64_t M, int64_t C) {
    const int64_t tiles = cdiv(C, 64);
    int64_t s = cdiv(2 * 148, tiles);
    s = s < 1 ? 1 : s;
    const int64_t maxs = cdiv(M, 64) < 1 ? 1 : cdiv(M, 64);
    s = s > maxs ? maxs : s;
    int64_t rows = up((size_t)cdiv(M, s), 64);
    if (rows < 64) rows = 64;
    return {rows, M > 0 ? cdiv(M, rows) : 1};
}

struct BwdWs {
    uint16_t *Bt, *sV, *U, *Bp, *Ap;
    float *part;
};
size_t bwd_ws(int64_t M, int64_t N, int64_t K, int r, void *ws, BwdWs *out) {
    const int r8 = (int)up(r, 8), rp = lora_pad(r);
    const bool tc = M >= kTcMinM && (N % 8) == 0;
    size_t part;
    if (tc) {
        part = std::max(std::max(sk_plan(M, N, rp).part_floats, sk_plan(M, K, rp).part_floats),
                        std::max(sk_plan(K, M, rp).part_floats, sk_plan(N, M, rp).part_floats));
        const GemmSplit g = gemm_split(M, K, cdiv(N, 64));
        if (g.splits > 1) part = std::max(part, (size_t)g.splits * M * K);
    } else {
        const GradSplit ga = grad_split(M, K), gb = grad_split(M, N);
        part = (size_t)r * (size_t)std::max(ga.nchunks * K, gb.nchunks * N);
    }
    Carve c(ws);
    uint16_t *Bt = c.take<uint16_t>(tc ? 0 : (size_t)r8 * N);
    uint16_t *sV = c.take<uint16_t>((size_t)M * rp);
    uint16_t *U = c.take<uint16_t>((size_t)M * rp);
    uint16_t *Bp = c.take<uint16_t>(tc ? (size_t)N * rp : 0);
    uint16_t *Ap = c.take<uint16_t>(tc ? (size_t)rp * K : 0);
    float *p = c.take<float>(part);
    if (out) *out = BwdWs{Bt, sV, U, Bp, Ap, p};
    return c.off;
}

// ---- tensor maps (driver entry point fetched through the runtime) ----------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// 2-D tiled map over a row-major [outer, inner] array (inner contiguous).
qlora_status make_map(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t outer,
                      uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw,
                      const char *what) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(QLORA_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(QLORA_ERR_CUDA, "tensor map for %s: error %d", what, (int)r);
    return QLORA_OK;
}

// Device check for the tcgen05 kernels (compiled for sm_103a only).
qlora_status tc_device_ok() {
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return fail(QLORA_ERR_CUDA, "cannot query the current device");
    if (major != 10 || minor != 3)
        return fail(QLORA_ERR_UNSUPPORTED, "device is sm_%d%d; this library is built for sm_103a", major, minor);
    return QLORA_OK;
}

template <int MODE>
qlora_status tc_setup() {
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        err = cudaFuncSetAttribute(k_gemm_tc<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg::SMEM_BYTES);
    });
    if (err != cudaSuccess) return fail(QLORA_ERR_CUDA, "setting shared memory size: %s", cudaGetErrorString(err));
    return QLORA_OK;
}

constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s per bounded wait
uint64_t wait_ns() { return g_wait_limit > 0 ? (uint64_t)g_wait_limit * 1000ull : kDefaultWaitNs; }

template <int A_MN, int B_MN>
qlora_status run_skinny(const CUtensorMap &ta, const CUtensorMap &tb, const SkPlan &pl, float *part, cudaStream_t s,
                        unsigned id) {
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        err = cudaFuncSetAttribute(k_gemm_skinny<A_MN, B_MN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   SkCfg::SMEM_BYTES);
    });
    if (err != cudaSuccess) return fail(QLORA_ERR_CUDA, "setting shared memory size: %s", cudaGetErrorString(err));
    SkParams prm{pl.rows, pl.rows_pad, pl.L, pl.spc, part, wait_ns(), id};
    dim3 grid((unsigned)(pl.rows_pad / 128), (unsigned)pl.chunks, (unsigned)pl.zt);
    {
        ProfScope ps(id == 5 || id == 6 ? QLORA_KERNEL_GRADS : QLORA_KERNEL_LORA_PRE, s);
        k_gemm_skinny<A_MN, B_MN><<<grid, SkCfg::THREADS, SkCfg::SMEM_BYTES, s>>>(ta, tb, prm);
    }
    return launch_check("k_gemm_skinny");
}

qlora_status run_reduce(const SkPlan &pl, const float *part, int r, int rp, float scale, int mode, uint16_t *o16a,
                        int lda, uint16_t *o16b, int ldb, float *o32, cudaStream_t s) {
    {
        ProfScope ps(mode >= kRedDA ? QLORA_KERNEL_GRADS : QLORA_KERNEL_LORA_PRE, s);
        k_skinny_reduce<<<(unsigned)cdiv(pl.rows * rp, 256), 256, 0, s>>>(part, (int)pl.chunks, pl.rows, pl.rows_pad,
                                                                         r, rp, scale, mode, o16a, lda, o16b, ldb,
                                                                         o32);
    }
    return launch_check("k_skinny_reduce");
}

}  // namespace

extern "C" {

const char *qlora_version(void) { return "qlora-b300 0.1 (sm_103a)"; }

const char *qlora_last_error(void) { return t_last_error.c_str(); }

void qlora_set_wait_limit(int64_t microseconds) { g_wait_limit = microseconds > 0 ? microseconds : 0; }

void qlora_nf4_table(float levels[16]) {
    static const float L[16] = QLORA_NF4_LEVELS;
    if (levels) memcpy(levels, L, sizeof L);
}

size_t qlora_nf4_codes_bytes(int64_t rows, int64_t cols) {
    return valid_dims(rows, cols) ? (size_t)(rows * cols / 2) : 0;
}
size_t qlora_nf4_absmax_count(int64_t rows, int64_t cols) {
    return valid_dims(rows, cols) ? (size_t)(rows * cols / kBlock) : 0;
}
size_t qlora_nf4_scale_count(int64_t rows, int64_t cols) {
    return valid_dims(rows, cols) ? (size_t)cdiv(rows * cols / kBlock, kGroup) : 0;
}
size_t qlora_nf4_storage_bytes(int64_t rows, int64_t cols) {
    if (!valid_dims(rows, cols)) return 0;
    return up(qlora_nf4_codes_bytes(rows, cols), 16) + up(qlora_nf4_absmax_count(rows, cols), 16) +
           up(qlora_nf4_scale_count(rows, cols) * 4, 16) + 16;
}
size_t qlora_nf4_quantize_workspace(int64_t rows, int64_t cols) {
    if (!valid_dims(rows, cols)) return 0;
    return quantize_ws(rows, cols, nullptr, nullptr, nullptr, nullptr, nullptr);
}

qlora_status qlora_nf4_quantize(const void *W, qlora_nf4_weight *out, void *ws, size_t ws_bytes,
                                qlora_stream_t stream) {
    qlora_status st = check_weight(out, false);
    if (st) return st;
    if (!W) return fail(QLORA_ERR_NULL, "W is NULL");
    if (!al16(W)) return fail(QLORA_ERR_ALIGN, "W must be 16-byte aligned");
    const int64_t rows = out->rows, cols = out->cols;
    if (rows == 0) return ok();
    if (!ws) return fail(QLORA_ERR_NULL, "workspace is NULL");
    if (!al16(ws)) return fail(QLORA_ERR_ALIGN, "workspace must be 16-byte aligned");
    float *absmax;
    double *gsum, *b0, *b1;
    const size_t need = quantize_ws(rows, cols, &absmax, &gsum, &b0, &b1, ws);
    if (ws_bytes < need)
        return fail(QLORA_ERR_WORKSPACE, "quantize workspace %zu < %zu bytes", ws_bytes, need);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t nb = rows * cols / kBlock, ng = cdiv(nb, kGroup);
    {
        ProfScope ps(QLORA_KERNEL_QUANTIZE, s);
        k_nf4_encode<<<(unsigned)ng, 256, 0, s>>>(static_cast<const uint4 *>(W), nb,
                                                 reinterpret_cast<uint32_t *>(out->codes), absmax, gsum);
    }
    if ((st = launch_check("k_nf4_encode"))) return st;
    // continue the pairwise tree over the group sums, 256 per warp
    const double *cur = gsum;
    int64_t n = ng;
    double *bufs[2] = {b0, b1};
    int flip = 0;
    while (n > 256) {
        const int64_t chunks = cdiv(n, 256);
        {
            ProfScope ps(QLORA_KERNEL_QUANTIZE, s);
            k_pairwise_reduce<<<(unsigned)cdiv(chunks, 8), 256, 0, s>>>(cur, n, bufs[flip], nullptr, nb);
        }
        if ((st = launch_check("k_pairwise_reduce"))) return st;
        cur = bufs[flip];
        flip ^= 1;
        n = chunks;
    }
    {
        ProfScope ps(QLORA_KERNEL_QUANTIZE, s);
        k_pairwise_reduce<<<1, 256, 0, s>>>(cur, n, nullptr, out->absmax_mean, nb);
    }
    if ((st = launch_check("k_pairwise_reduce(mean)"))) return st;
    {
        ProfScope ps(QLORA_KERNEL_QUANTIZE, s);
        k_dq_encode<<<(unsigned)cdiv(ng, 8), 256, 0, s>>>(absmax, nb, out->absmax_mean, out->absmax_q,
                                                          out->absmax_scale);
    }
    if ((st = launch_check("k_dq_encode"))) return st;
    return ok();
}

// ---- quantize without a caller workspace ------------------------------------
// The scratch lives in this file-scope device array. In host code its name is
// only a host-side stand-in, so the device address is looked up with
// cudaGetSymbolAddress, once per device, with that device current.
static __device__ __align__(256) unsigned char g_quantize_scratch[QLORA_NF4_NOALLOC_SCRATCH_BYTES];
static std::mutex g_scratch_mu;
static void *g_scratch_ptr[128] = {};

static qlora_status quantize_scratch(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(QLORA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 128) return fail(QLORA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_quantize_scratch);
        if (e != cudaSuccess || !p)
            return fail(QLORA_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return QLORA_OK;
}

qlora_status qlora_nf4_quantize_noalloc(const void *W, qlora_nf4_weight *out, qlora_stream_t stream) {
    qlora_status st = check_weight(out, false);
    if (st) return st;
    if (!W) return fail(QLORA_ERR_NULL, "W is NULL");
    if (!al16(W)) return fail(QLORA_ERR_ALIGN, "W must be 16-byte aligned");
    const int64_t rows = out->rows, cols = out->cols;
    if (rows == 0) return ok();
    const size_t need = quantize_ws(rows, cols, nullptr, nullptr, nullptr, nullptr, nullptr);
    if (need > QLORA_NF4_NOALLOC_SCRATCH_BYTES)
        return fail(QLORA_ERR_WORKSPACE,
                    "weight [%lld, %lld] needs %zu bytes of scratch; the built-in scratch holds %u bytes "
                    "(use qlora_nf4_quantize with a workspace)",
                    (long long)rows, (long long)cols, need, QLORA_NF4_NOALLOC_SCRATCH_BYTES);
    void *scratch = nullptr;
    if ((st = quantize_scratch(&scratch))) return st;
    float *absmax;
    double *gsum, *b0, *b1;
    quantize_ws(rows, cols, &absmax, &gsum, &b0, &b1, scratch);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t nb = rows * cols / kBlock, ng = cdiv(nb, kGroup);
    k_nf4_encode<<<(unsigned)ng, 256, 0, s>>>(static_cast<const uint4 *>(W), nb,
                                             reinterpret_cast<uint32_t *>(out->codes), absmax, gsum);
    if ((st = launch_check("k_nf4_encode"))) return st;
    const double *cur = gsum;
    int64_t n = ng;
    double *bufs[2] = {b0, b1};
    int flip = 0;
    while (n > 256) {
        const int64_t chunks = cdiv(n, 256);
        k_pairwise_reduce<<<(unsigned)cdiv(chunks, 8), 256, 0, s>>>(cur, n, bufs[flip], nullptr, nb);
        if ((st = launch_check("k_pairwise_reduce"))) return st;
        cur = bufs[flip];
        flip ^= 1;
        n = chunks;
    }
    k_pairwise_reduce<<<1, 256, 0, s>>>(cur, n, nullptr, out->absmax_mean, nb);
    if ((st = launch_check("k_pairwise_reduce(mean)"))) return st;
    k_dq_encode<<<(unsigned)cdiv(ng, 8), 256, 0, s>>>(absmax, nb, out->absmax_mean, out->absmax_q,
                                                      out->absmax_scale);
    if ((st = launch_check("k_dq_encode"))) return st;
    return ok();
}

qlora_status qlora_nf4_dequantize(const qlora_nf4_weight *w, void *out, qlora_stream_t stream) {
    qlora_status st = check_weight(w, false);
    if (st) return st;
    if (!out) return fail(QLORA_ERR_NULL, "output is NULL");
    if (!al16(out)) return fail(QLORA_ERR_ALIGN, "output must be 16-byte aligned");
    if (w->rows == 0) return ok();
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t nhalf = w->rows * w->cols / 32;
    {
        ProfScope ps(QLORA_KERNEL_DEQUANT, s);
        k_nf4_dequant<<<(unsigned)cdiv(nhalf, 256), 256, 0, s>>>(reinterpret_cast<const uint4 *>(w->codes),
                                                                 w->absmax_q, w->absmax_scale, w->absmax_mean,
                                                                 nhalf, static_cast<uint4 *>(out));
    }
    if ((st = launch_check("k_nf4_dequant"))) return st;
    return ok();
}

size_t qlora_linear_fwd_workspace(int64_t M, const qlora_nf4_weight *w, int r) {
    if (!w || !valid_dims(w->rows, w->cols) || M < 0 || r < 1 || r > 128) return 0;
    return fwd_ws(M, w->rows, w->cols, r, nullptr, nullptr);
}

size_t qlora_linear_bwd_workspace(int64_t M, const qlora_nf4_weight *w, int r) {
    if (!w || !valid_dims(w->rows, w->cols) || M < 0 || r < 1 || r > 128) return 0;
    return bwd_ws(M, w->rows, w->cols, r, nullptr, nullptr);
}

static qlora_status check_linear_common(int64_t M, const qlora_nf4_weight *w, const void *A, const void *B, int r,
                                        void *ws) {
    qlora_status st = check_weight(w, true);
    if (st) return st;
    if (M < 0 || M >= kMaxDim) return fail(QLORA_ERR_SHAPE, "M = %lld out of range", (long long)M);
    if (r < 1 || r > 128) return fail(QLORA_ERR_RANK, "LoRA rank r = %d outside [1, 128]", r);
    if (!A || !B) return fail(QLORA_ERR_NULL, "LoRA A or B is NULL");
    if (!al16(A) || !al16(B)) return fail(QLORA_ERR_ALIGN, "LoRA A and B must be 16-byte aligned");
    if (ws && !al16(ws)) return fail(QLORA_ERR_ALIGN, "workspace must be 16-byte aligned");
    return QLORA_OK;
}

qlora_status qlora_linear_fwd(const void *X, int64_t M, const qlora_nf4_weight *w, const void *A, const void *B,
                              int r, float scale, void *Y, void *U_save, void *ws, size_t ws_bytes,
                              qlora_stream_t stream) {
    qlora_status st = check_linear_common(M, w, A, B, r, ws);
    if (st) return st;
    if (M > 0 && (!X || !Y)) return fail(QLORA_ERR_NULL, "X or Y is NULL");
    if ((X && !al16(X)) || (Y && !al16(Y)) || (U_save && !al16(U_save)))
        return fail(QLORA_ERR_ALIGN, "X, Y and U_save must be 16-byte aligned");
    if (M == 0) return ok();
    const int64_t N = w->rows, K = w->cols;
    FwdWs f;
    const size_t need = fwd_ws(M, N, K, r, ws, &f);
    if (!ws) return fail(QLORA_ERR_NULL, "workspace is NULL");
    if (ws_bytes < need) return fail(QLORA_ERR_WORKSPACE, "forward workspace %zu < %zu bytes", ws_bytes, need);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int rp = lora_pad(r);
    const uint16_t *X16 = static_cast<const uint16_t *>(X);
    uint16_t *U16 = static_cast<uint16_t *>(U_save);

    if (M < kTcMinM) {
        // small M: CUDA-core kernels
        {
            ProfScope ps(QLORA_KERNEL_LORA_PRE, s);
            k_lora_down<<<(unsigned)cdiv(M, 16), 256, 0, s>>>(X16, M, K, static_cast<const uint16_t *>(A), r, scale,
                                                              U16, r, f.sU, rp);
        }
        if ((st = launch_check("k_lora_down"))) return st;
        dim3 grid((unsigned)cdiv(N, kSt), (unsigned)cdiv(M, kSt));
        {
            ProfScope ps(QLORA_KERNEL_FWD_SIMT, s);
            k_fwd_simt<<<grid, 256, 0, s>>>(X16, M, K, w->codes, w->absmax_q, w->absmax_scale, w->absmax_mean, N,
                                            f.sU, rp, static_cast<const uint16_t *>(B), r,
                                            static_cast<uint16_t *>(Y));
        }
        if ((st = launch_check("k_fwd_simt"))) return st;
        return ok();
    }

    if ((st = tc_device_ok()) || (st = tc_setup<kFwd>())) return st;
    {
        ProfScope ps(QLORA_KERNEL_LORA_PRE, s);
        k_pad_rows<<<(unsigned)cdiv(rp * K, 256), 256, 0, s>>>(static_cast<const uint16_t *>(A), r, rp, K, f.Ap);
    }
    if ((st = launch_check("k_pad_rows(A)"))) return st;
    {
        ProfScope ps(QLORA_KERNEL_LORA_PRE, s);
        k_pad_cols<<<(unsigned)cdiv(N * rp, 256), 256, 0, s>>>(static_cast<const uint16_t *>(B), N, r, rp, f.Bp);
    }
    if ((st = launch_check("k_pad_cols(B)"))) return st;
    CUtensorMap tmX, tmC, tmU, tmB, tmA;
    if ((st = make_map(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, K, M, K * 2, 64, 128,
                       CU_TENSOR_MAP_SWIZZLE_128B, "X")) ||
        (st = make_map(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, f.Ap, K, rp, K * 2, 64, 64,
                       CU_TENSOR_MAP_SWIZZLE_128B, "A")) ||
        (st = make_map(&tmC, CU_TENSOR_MAP_DATA_TYPE_UINT8, w->codes, K / 2, N, K / 2, 32, 256,
                       CU_TENSOR_MAP_SWIZZLE_32B, "codes")) ||
        (st = make_map(&tmU, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, f.sU, rp, M, rp * 2, 64, 128,
                       CU_TENSOR_MAP_SWIZZLE_128B, "sU")) ||
        (st = make_map(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, f.Bp, rp, N, rp * 2, 64, 256,
                       CU_TENSOR_MAP_SWIZZLE_128B, "B")))
        return st;
    // U = X A^T on the tensor cores; U (bf16) to U_save, s*U (bf16) to the workspace
    const SkPlan pu = sk_plan(M, K, rp);
    if ((st = run_skinny<0, 0>(tmX, tmA, pu, f.part, s, 3))) return st;
    if ((st = run_reduce(pu, f.part, r, rp, scale, kRedU, U16, r, f.sU, rp, nullptr, s))) return st;
    TcParams prm{};
    prm.M = M;
    prm.Nd = N;
    prm.w_rows = N;
    prm.w_cols = K;
    prm.nk_main = K / TcCfg::BK;
    prm.lora_steps = rp / 64;
    prm.r = r;
    prm.q = w->absmax_q;
    prm.s2 = w->absmax_scale;
    prm.mean = w->absmax_mean;
    prm.out = static_cast<uint16_t *>(Y);
    prm.ldo = N;
    const GemmSplit gs = gemm_split(M, N, prm.nk_main);
    prm.splits = gs.splits;
    prm.steps_per_split = gs.steps_per_split;
    prm.part = f.part;
    prm.wait_ns = wait_ns();
    prm.kernel_id = 1;
    dim3 grid((unsigned)cdiv(N, TcCfg::BN), (unsigned)cdiv(M, TcCfg::BM), (unsigned)gs.splits);
    {
        ProfScope ps(QLORA_KERNEL_FWD_GEMM, s);
        k_gemm_tc<kFwd><<<grid, TcCfg::THREADS, TcCfg::SMEM_BYTES, s>>>(tmX, tmC, tmU, tmB, prm);
    }
    if ((st = launch_check("k_gemm_tc<fwd>"))) return st;
    if (gs.splits > 1) {
        {
            ProfScope ps(QLORA_KERNEL_FWD_GEMM, s);
            k_split_reduce<<<(unsigned)cdiv(cdiv(M * N, 4), 256), 256, 0, s>>>(f.part, gs.splits, M, N,
                                                                             static_cast<uint16_t *>(Y), N);
        }
        if ((st = launch_check("k_split_reduce"))) return st;
    }
    return ok();
}

qlora_status qlora_linear_bwd(const void *dY, const void *X, const void *U_saved, int64_t M,
                              const qlora_nf4_weight *w, const void *A, const void *B, int r, float scale, void *dX,
                              float *dA, float *dB, void *ws, size_t ws_bytes, qlora_stream_t stream) {
    qlora_status st = check_linear_common(M, w, A, B, r, ws);
    if (st) return st;
    if (!dA || !dB) return fail(QLORA_ERR_NULL, "dA or dB is NULL");
    if (M > 0 && (!dY || !X || !dX)) return fail(QLORA_ERR_NULL, "dY, X or dX is NULL");
    if ((dY && !al16(dY)) || (X && !al16(X)) || (dX && !al16(dX)) || !al16(dA) || !al16(dB) ||
        (U_saved && !al16(U_saved)))
        return fail(QLORA_ERR_ALIGN, "dY, X, U_saved, dX, dA and dB must be 16-byte aligned");
    const int64_t N = w->rows, K = w->cols;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (M == 0) {
        if (cudaMemsetAsync(dA, 0, sizeof(float) * r * K, s) != cudaSuccess ||
            cudaMemsetAsync(dB, 0, sizeof(float) * r * N, s) != cudaSuccess)
            return fail(QLORA_ERR_CUDA, "memset of dA/dB failed");
        return ok();
    }
    BwdWs b;
    const size_t need = bwd_ws(M, N, K, r, ws, &b);
    if (!ws) return fail(QLORA_ERR_NULL, "workspace is NULL");
    if (ws_bytes < need) return fail(QLORA_ERR_WORKSPACE, "backward workspace %zu < %zu bytes", ws_bytes, need);
    const int r8 = (int)up(r, 8), rp = lora_pad(r);
    const uint16_t *dY16 = static_cast<const uint16_t *>(dY), *X16 = static_cast<const uint16_t *>(X);
    const uint16_t *A16 = static_cast<const uint16_t *>(A), *B16 = static_cast<const uint16_t *>(B);
    const bool tc = M >= kTcMinM && (N % 8) == 0;

    if (!tc) {
        // small M (or N not a multiple of 8): CUDA-core kernels
        {
            ProfScope ps(QLORA_KERNEL_LORA_PRE, s);
            k_transpose<<<(unsigned)cdiv(N, 256), 256, 0, s>>>(B16, N, r, r8, b.Bt);
        }
        if ((st = launch_check("k_transpose"))) return st;
        {
            ProfScope ps(QLORA_KERNEL_LORA_PRE, s);
            k_lora_down<<<(unsigned)cdiv(M, 16), 256, 0, s>>>(dY16, M, N, b.Bt, r, scale, nullptr, 0, b.sV, rp);
        }
        if ((st = launch_check("k_lora_down(V)"))) return st;
        const uint16_t *U = static_cast<const uint16_t *>(U_saved);
        int ldu = r;
        if (!U) {
            {
                ProfScope ps(QLORA_KERNEL_LORA_PRE, s);
                k_lora_down<<<(unsigned)cdiv(M, 16), 256, 0, s>>>(X16, M, K, A16, r, 1.0f, nullptr, 0, b.U, rp);
            }
            if ((st = launch_check("k_lora_down(U)"))) return st;
            U = b.U;
            ldu = rp;
        }
        dim3 grid((unsigned)cdiv(K, kSt), (unsigned)cdiv(M, kSt));
        {
            ProfScope ps(QLORA_KERNEL_DX_SIMT, s);
            k_dx_simt<<<grid, 256, 0, s>>>(dY16, M, N, w->codes, w->absmax_q, w->absmax_scale, w->absmax_mean, K,
                                           b.sV, rp, A16, r, static_cast<uint16_t *>(dX));
        }
        if ((st = launch_check("k_dx_simt"))) return st;
        GradSplit ga = grad_split(M, K);
        {
            ProfScope ps(QLORA_KERNEL_GRADS, s);
            k_lora_grad<<<dim3((unsigned)cdiv(K, 64), (unsigned)ga.nchunks), 256, 0, s>>>(b.sV, rp, X16, M, K, r,
                                                                                       ga.rows_per_chunk, b.part);
        }
        if ((st = launch_check("k_lora_grad(dA)"))) return st;
        {
            ProfScope ps(QLORA_KERNEL_GRADS, s);
            k_grad_reduce<<<(unsigned)cdiv((int64_t)r * K, 256), 256, 0, s>>>(b.part, (int)ga.nchunks, r, K, 1.0f,
                                                                              0, dA);
        }
        if ((st = launch_check("k_grad_reduce(dA)"))) return st;
        GradSplit gb = grad_split(M, N);
        {
            ProfScope ps(QLORA_KERNEL_GRADS, s);
            k_lora_grad<<<dim3((unsigned)cdiv(N, 64), (unsigned)gb.nchunks), 256, 0, s>>>(U, ldu, dY16, M, N, r,
                                                                                       gb.rows_per_chunk, b.part);
        }
        if ((st = launch_check("k_lora_grad(dB)"))) return st;
        {
            ProfScope ps(QLORA_KERNEL_GRADS, s);
            k_grad_reduce<<<(unsigned)cdiv((int64_t)r * N, 256), 256, 0, s>>>(b.part, (int)gb.nchunks, r, N, scale,
                                                                              1, dB);
        }
        if ((st = launch_check("k_grad_reduce(dB)"))) return st;
        return ok();
    }

    if ((st = tc_device_ok()) || (st = tc_setup<kDx>())) return st;
    {
        ProfScope ps(QLORA_KERNEL_LORA_PRE, s);
        k_pad_cols<<<(unsigned)cdiv(N * rp, 256), 256, 0, s>>>(B16, N, r, rp, b.Bp);
    }
    if ((st = launch_check("k_pad_cols(B)"))) return st;
    {
        ProfScope ps(QLORA_KERNEL_LORA_PRE, s);
        k_pad_rows<<<(unsigned)cdiv(rp * K, 256), 256, 0, s>>>(A16, r, rp, K, b.Ap);
    }
    if ((st = launch_check("k_pad_rows(A)"))) return st;
    CUtensorMap tmD, tmDmn, tmXk, tmXmn, tmC, tmV, tmA, tmBp, tmUp;
    if ((st = make_map(&tmD, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dY, N, M, N * 2, 64, 128,
                       CU_TENSOR_MAP_SWIZZLE_128B, "dY")) ||
        (st = make_map(&tmDmn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dY, N, M, N * 2, 64, 64,
                       CU_TENSOR_MAP_SWIZZLE_128B, "dY (MN)")) ||
        (st = make_map(&tmXk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, K, M, K * 2, 64, 128,
                       CU_TENSOR_MAP_SWIZZLE_128B, "X")) ||
        (st = make_map(&tmXmn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, K, M, K * 2, 64, 64,
                       CU_TENSOR_MAP_SWIZZLE_128B, "X (MN)")) ||
        (st = make_map(&tmC, CU_TENSOR_MAP_DATA_TYPE_UINT8, w->codes, K / 2, N, K / 2, 128, 64,
                       CU_TENSOR_MAP_SWIZZLE_128B, "codes")) ||
        (st = make_map(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, b.sV, rp, M, rp * 2, 64, 128,
                       CU_TENSOR_MAP_SWIZZLE_128B, "sV")) ||
        (st = make_map(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, b.Ap, K, rp, K * 2, 64, 64,
                       CU_TENSOR_MAP_SWIZZLE_128B, "A")) ||
        (st = make_map(&tmBp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, b.Bp, rp, N, rp * 2, 64, 64,
                       CU_TENSOR_MAP_SWIZZLE_128B, "B")) ||
        (st = make_map(&tmUp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, b.U, rp, M, rp * 2, 64, 64,
                       CU_TENSOR_MAP_SWIZZLE_128B, "U")))
        return st;
    CUtensorMap tmVmn;
    if ((st = make_map(&tmVmn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, b.sV, rp, M, rp * 2, 64, 64,
                       CU_TENSOR_MAP_SWIZZLE_128B, "sV (MN)")))
        return st;
    // V = dY B -> sV = bf16(s * V)
    const SkPlan pv = sk_plan(M, N, rp);
    if ((st = run_skinny<0, 1>(tmD, tmBp, pv, b.part, s, 4))) return st;
    if ((st = run_reduce(pv, b.part, r, rp, scale, kRedV, nullptr, 0, b.sV, rp, nullptr, s))) return st;
    // U (padded to rp columns): from the forward's U, or recomputed as X A^T
    if (U_saved) {
        ProfScope ps(QLORA_KERNEL_LORA_PRE, s);
        k_pad_cols<<<(unsigned)cdiv(M * rp, 256), 256, 0, s>>>(static_cast<const uint16_t *>(U_saved), M, r, rp, b.U);
    } else {
        const SkPlan pu = sk_plan(M, K, rp);
        if ((st = run_skinny<0, 0>(tmXk, tmA, pu, b.part, s, 3))) return st;
        if ((st = run_reduce(pu, b.part, r, rp, 1.0f, kRedU, nullptr, 0, b.U, rp, nullptr, s))) return st;
    }
    if ((st = launch_check("U"))) return st;
    // dX = dY W' + (sV) A
    TcParams prm{};
    prm.M = M;
    prm.Nd = K;
    prm.w_rows = N;
    prm.w_cols = K;
    prm.nk_main = cdiv(N, TcCfg::BK);
    prm.lora_steps = rp / 64;
    prm.r = r;
    prm.q = w->absmax_q;
    prm.s2 = w->absmax_scale;
    prm.mean = w->absmax_mean;
    prm.out = static_cast<uint16_t *>(dX);
    prm.ldo = K;
    const GemmSplit gs = gemm_split(M, K, prm.nk_main);
    prm.splits = gs.splits;
    prm.steps_per_split = gs.steps_per_split;
    prm.part = b.part;
    prm.wait_ns = wait_ns();
    prm.kernel_id = 2;
    {
        dim3 grid((unsigned)cdiv(K, TcCfg::BN), (unsigned)cdiv(M, TcCfg::BM), (unsigned)gs.splits);
        ProfScope ps(QLORA_KERNEL_DX_GEMM, s);
        k_gemm_tc<kDx><<<grid, TcCfg::THREADS, TcCfg::SMEM_BYTES, s>>>(tmD, tmC, tmV, tmA, prm);
    }
    if ((st = launch_check("k_gemm_tc<dx>"))) return st;
    if (gs.splits > 1) {
        {
            ProfScope ps(QLORA_KERNEL_DX_GEMM, s);
            k_split_reduce<<<(unsigned)cdiv(cdiv(M * K, 4), 256), 256, 0, s>>>(b.part, gs.splits, M, K,
                                                                             static_cast<uint16_t *>(dX), K);
        }
        if ((st = launch_check("k_split_reduce"))) return st;
    }
    // dA = (sV)^T X   (rows k of dA^T, contraction over the M tokens)
    const SkPlan pa = sk_plan(K, M, rp);
    if ((st = run_skinny<1, 1>(tmXmn, tmVmn, pa, b.part, s, 5))) return st;
    if ((st = run_reduce(pa, b.part, r, rp, 1.0f, kRedDA, nullptr, 0, nullptr, 0, dA, s))) return st;
    // dB = s dY^T U
    const SkPlan pb = sk_plan(N, M, rp);
    if ((st = run_skinny<1, 1>(tmDmn, tmUp, pb, b.part, s, 6))) return st;
    if ((st = run_reduce(pb, b.part, r, rp, scale, kRedDB, nullptr, 0, nullptr, 0, dB, s))) return st;
    return ok();
}

void qlora_profile_start(void) {
    for (auto &p : g_prof) {
        cudaEventDestroy(p.a);
        cudaEventDestroy(p.b);
    }
    g_prof.clear();
    for (int k = 0; k < QLORA_KERNEL_KINDS; ++k) g_prof_count[k] = 0;
    g_prof_on = true;
}

int qlora_profile_stop(double ms_per_kind[QLORA_KERNEL_KINDS], int launches_per_kind[QLORA_KERNEL_KINDS]) {
    g_prof_on = false;
    int total = 0, bad = 0;
    for (int k = 0; k < QLORA_KERNEL_KINDS; ++k) {
        if (ms_per_kind) ms_per_kind[k] = 0.0;
        if (launches_per_kind) launches_per_kind[k] = g_prof_count[k];
        total += g_prof_count[k];
    }
    for (auto &p : g_prof) {
        float ms = 0.0f;
        if (cudaEventSynchronize(p.b) != cudaSuccess || cudaEventElapsedTime(&ms, p.a, p.b) != cudaSuccess) bad = 1;
        if (ms_per_kind) ms_per_kind[p.kind] += ms;
        cudaEventDestroy(p.a);
        cudaEventDestroy(p.b);
    }
    g_prof.clear();
    return bad ? -1 : total;
}

qlora_status qlora_check_device_status(qlora_stream_t stream) {
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(QLORA_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
    unsigned int word = 0;
    e = cudaMemcpyFromSymbol(&word, g_error_word, sizeof word);
    if (e != cudaSuccess) return fail(QLORA_ERR_CUDA, "reading the device error word: %s", cudaGetErrorString(e));
    if (word) {
        const unsigned int zero = 0;
        cudaMemcpyToSymbol(g_error_word, &zero, sizeof zero);
        return fail(QLORA_ERR_TIMEOUT, "bounded wait ran out: kernel %u, site %u", word >> 16, word & 0xFFFFu);
    }
    return ok();
}

}  // extern "C"
