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
#include <array>

#include "qlora.h"

#include "common.cuh"
#include "codec.cuh"
#include "lora_simt.cuh"
#include "gemm_tc.cuh"
#include "gemm_pair.cuh"
#include "lora_tc.cuh"
#include "small_m.cuh"
#include "fwd_few.cuh"
#include "merge.cuh"
#include "adamw.cuh"

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

// Sets a kernel's dynamic shared memory limit once per (kernel, device): the
// attribute belongs to the device that is current when it is set.
std::mutex g_attr_mu;
std::vector<std::pair<const void *, int>> g_attr_done;

template <class Kern>
cudaError_t smem_attr(Kern kern, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const void *key = reinterpret_cast<const void *>(kern);
    std::lock_guard<std::mutex> lock(g_attr_mu);
    for (const auto &d : g_attr_done)
        if (d.first == key && d.second == dev) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) g_attr_done.push_back({key, dev});
    return e;
}

int current_device() {
    int dev = 0;
    return cudaGetDevice(&dev) == cudaSuccess ? dev : -1;
}

bool valid_dims(int64_t rows, int64_t cols) {
    return rows >= 0 && cols > 0 && cols % kBlock == 0 && rows < kMaxDim && cols < kMaxDim;
}

// Internal view of a quantized weight, from either descriptor of the ABI:
// the level table, and the block absmax either double-quantized (q, s2, mean)
// or as fp32 (absmax; then q, s2, mean are null).
struct Wt {
    int64_t rows, cols;
    int tab;
    uint8_t *codes;
    int8_t *q;
    float *s2, *mean;
    float *absmax;
    bool valid_format;
};
Wt wt_of(const qlora_nf4_weight *w) {
    return Wt{w->rows, w->cols, kTableNF4, w->codes, w->absmax_q, w->absmax_scale, w->absmax_mean, nullptr, true};
}
Wt wt_of(const qlora_q4_weight *w) {
    Wt t{w->rows, w->cols, w->table, w->codes, nullptr, nullptr, nullptr, nullptr, true};
    if (w->double_quant) {
        t.q = w->absmax_q;
        t.s2 = w->absmax_scale;
        t.mean = w->absmax_mean;
    } else {
        t.absmax = w->absmax;
    }
    t.valid_format = (w->table == kTableNF4 || w->table == kTableINT4) && (w->double_quant == 0 || w->double_quant == 1);
    return t;
}

qlora_status check_weight(const Wt &w, bool need_rows) {
    if (!w.valid_format) return fail(QLORA_ERR_UNSUPPORTED, "unknown table or double_quant value");
    if (!valid_dims(w.rows, w.cols))
        return fail(QLORA_ERR_SHAPE, "weight shape [%lld, %lld]: need rows >= 0, cols > 0, cols %% 64 == 0",
                    (long long)w.rows, (long long)w.cols);
    if (need_rows && w.rows == 0) return fail(QLORA_ERR_SHAPE, "weight has 0 rows");
    if (!w.codes || (w.absmax ? false : (!w.q || !w.s2 || !w.mean)) || (!w.q && !w.absmax))
        return fail(QLORA_ERR_NULL, "weight descriptor has a NULL array");
    if (!al16(w.codes) || (w.absmax && !al16(w.absmax)) || (w.q && (!al16(w.q) || !al16(w.s2) || !al16(w.mean))))
        return fail(QLORA_ERR_ALIGN, "weight arrays must be 16-byte aligned");
    return QLORA_OK;
}
qlora_status check_weight(const qlora_nf4_weight *w, bool need_rows) {
    if (!w) return fail(QLORA_ERR_NULL, "weight descriptor is NULL");
    return check_weight(wt_of(w), need_rows);
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

// The quantizer's launch sequence on a carved scratch area (the caller's
// workspace or the built-in array): encode with the exact absmax and the
// group sums of the pairwise tree, the tree's upper levels 256 values at a
// time down to the mean, then the int8 codes and group scales.
qlora_status quantize_launch(const void *W, const Wt &out, float *absmax, double *gsum, double *b0,
                             double *b1, cudaStream_t s) {
    const int64_t nb = out.rows * out.cols / kBlock, ng = cdiv(nb, kGroup);
    qlora_status st;
    if (out.absmax) {
        // no double quantization: the exact block absmax is the stored constant
        ProfScope ps(QLORA_KERNEL_QUANTIZE, s);
        k_nf4_encode<<<(unsigned)ng, 256, 0, s>>>(static_cast<const uint4 *>(W), nb,
                                                 reinterpret_cast<uint32_t *>(out.codes), out.absmax, nullptr,
                                                 out.tab);
        return launch_check("k_nf4_encode");
    }
    {
        ProfScope ps(QLORA_KERNEL_QUANTIZE, s);
        k_nf4_encode<<<(unsigned)ng, 256, 0, s>>>(static_cast<const uint4 *>(W), nb,
                                                 reinterpret_cast<uint32_t *>(out.codes), absmax, gsum, out.tab);
    }
    if ((st = launch_check("k_nf4_encode"))) return st;
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
        k_pairwise_reduce<<<1, 256, 0, s>>>(cur, n, nullptr, out.mean, nb);
    }
    if ((st = launch_check("k_pairwise_reduce(mean)"))) return st;
    {
        ProfScope ps(QLORA_KERNEL_QUANTIZE, s);
        k_dq_encode<<<(unsigned)cdiv(ng, 8), 256, 0, s>>>(absmax, nb, out.mean, out.q, out.s2);
    }
    if ((st = launch_check("k_dq_encode"))) return st;
    return ok();
}

// ---- linear workspaces
// Small-M (CUDA-core) path: the LoRA operands sU / sV / U are kept with rows
// of rp = 64 * ceil(r / 64) columns.
inline int lora_pad(int r) { return (int)up((size_t)r, 64); }
// Tensor-core path: sU / sV / U rows of rs = 8 * ceil(r / 8) columns (16-byte
// rows for TMA); the TMA zero fill supplies the rank padding up to 64.
inline int lora_rs(int r) { return (int)up((size_t)r, 8); }

// Tokens at or above which the tensor-core path runs.
constexpr int64_t kTcMinM = 64;

// One skinny tcgen05 pass (k_lora_skinny): output rows in 128-row tiles,
// rank in 64-wide tiles; the contraction is split into `chunks` (one cluster
// per tile), chosen at launch (see skinny_chunks).
struct SkPlan {
    int64_t rows, L, spc, chunks, tiles;
    int zt;
};
SkPlan sk_plan(int64_t rows, int64_t L, int r) {
    SkPlan p;
    p.rows = rows;
    p.tiles = cdiv(rows, 128);
    p.L = L;
    p.zt = (r + 63) / 64;
    p.spc = std::max<int64_t>(1, cdiv(L, 64));
    p.chunks = 1;
    return p;
}

// Stream-K hand-off area of the fused GEMM: the ready flags and arrival
// counters (zeroed by the skinny kernel that precedes the GEMM in the same
// call) and two fp32 partial-tile slots per CTA pair.
struct SkArea {
    uint32_t *flags;
    float *slots;
};
SkArea take_sk_area(Carve &c) {
    SkArea a;
    a.flags = c.take<uint32_t>((size_t)kSkFlagWords);
    // 32-byte stores into the slots: align within the (16-byte aligned) workspace
    char *raw = c.take<char>((size_t)kSkPairs * 2 * (size_t)kSlotFloats * sizeof(float) + 32);
    a.slots = raw ? reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(raw) + 31) & ~uintptr_t(31)) : nullptr;
    return a;
}

// The few-token forward (k_fwd_few) serves M <= 16 when K is a multiple of
// its 256-deep tasks (and the block count fits 31 bits); other few-token
// shapes take k_fwd_small.
inline bool few_path(int64_t M, int64_t N, int64_t K) {
    return M <= 8 * FewCfg::MAX_NT && K % FewCfg::TK == 0 && N * (K / kBlock) < (int64_t(1) << 31);
}

// Its split: tasks of 32 rows x 256 k over the warps of at most 148 CTAs
// (16 warps a CTA for M <= 8, 12 for two 8-token tiles), every warp at least
// one task.
struct FewPlan {
    int64_t grid, warps, tasks, tpr, tiles, wpc;
};
// tiles: the 32-row tiles of all the launch's projections
FewPlan few_plan_tiles(int64_t M, int64_t tiles, int64_t K) {
    FewPlan f;
    f.wpc = M <= 8 ? few_warps<1>() : few_warps<2>();
    f.tiles = tiles;
    f.tpr = K / FewCfg::TK;
    f.tasks = f.tiles * f.tpr;
    f.warps = std::min<int64_t>(f.tasks, f.wpc * FewCfg::GRID);
    f.grid = cdiv(f.warps, f.wpc);
    return f;
}
FewPlan few_plan(int64_t M, int64_t N, int64_t K) { return few_plan_tiles(M, cdiv(N, FewCfg::ROWS), K); }
// fp32 slot floats per warp: two row tiles x 32 lanes x 8 per 8-token tile
inline size_t few_slot_floats(int64_t M) { return (size_t)2 * 32 * 8 * (M <= 8 ? 1 : 2); }

struct FwdWs {
    uint16_t *sU, *Bp;
    float *few_slots;
    uint32_t *few_counters;
    SkArea sk;
};
size_t fwd_ws(int64_t M, int64_t N, int64_t K, int r, void *ws, FwdWs *out) {
    const bool tc = M > kSmallMaxM || K > kSmallMaxK;
    Carve c(ws);
    FwdWs f{};
    if (few_path(M, N, K)) {
        const FewPlan fp = few_plan(M, N, K);
        f.sU = c.take<uint16_t>((size_t)M * lora_pad(r));
        f.few_slots = c.take<float>((size_t)fp.warps * few_slot_floats(M));
        f.few_counters = c.take<uint32_t>((size_t)fp.tiles);
    } else if (!tc) {
        f.sU = c.take<uint16_t>((size_t)M * lora_pad(r));
    } else {
        const int rs = lora_rs(r);
        f.sU = c.take<uint16_t>((size_t)M * rs);
        f.Bp = c.take<uint16_t>(r % 8 ? (size_t)N * rs : 0);
        f.sk = take_sk_area(c);
    }
    if (out) *out = f;
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
    uint16_t *Bt, *sV, *U, *Bp;
    float *part;  // CUDA-core path: per-chunk adapter-gradient partials
    SkArea sk;
};
size_t bwd_ws(int64_t M, int64_t N, int64_t K, int r, void *ws, BwdWs *out) {
    const int r8 = (int)up(r, 8), rp = lora_pad(r), rs = lora_rs(r);
    const bool tc = M >= kTcMinM && (N % 8) == 0;
    Carve c(ws);
    BwdWs b{};
    if (!tc) {
        const GradSplit ga = grad_split(M, K), gb = grad_split(M, N);
        b.Bt = c.take<uint16_t>((size_t)r8 * N);
        b.sV = c.take<uint16_t>((size_t)M * rp);
        b.U = c.take<uint16_t>((size_t)M * rp);
        b.part = c.take<float>((size_t)r * (size_t)std::max(ga.nchunks * K, gb.nchunks * N));
    } else {
        b.sV = c.take<uint16_t>((size_t)M * rs);
        b.U = c.take<uint16_t>((size_t)M * rs);
        b.Bp = c.take<uint16_t>(r % 8 ? (size_t)N * rs : 0);
        b.sk = take_sk_area(c);
    }
    if (out) *out = b;
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
    const cudaError_t err = smem_attr(k_gemm_pair<MODE>, PairCfg::SMEM_BYTES);
    if (err != cudaSuccess) return fail(QLORA_ERR_CUDA, "setting shared memory size: %s", cudaGetErrorString(err));
    return QLORA_OK;
}

// Pairs of the persistent fused GEMM that the current device holds at once
// (queried once per device; the kernel's attribute is set by tc_setup first).
template <int MODE>
int64_t gemm_pairs_resident() {
    static std::mutex mu;
    static std::vector<std::pair<int, int>> cache;  // (device, clusters)
    const int dev = current_device();
    std::lock_guard<std::mutex> lock(mu);
    int n = -1;
    for (const auto &c : cache)
        if (c.first == dev) n = c.second;
    if (n < 0) {
        n = 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2, 1, 1);
        cfg.blockDim = dim3(PairCfg::THREADS);
        cfg.dynamicSmemBytes = PairCfg::SMEM_BYTES;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, k_gemm_pair<MODE>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        cache.push_back({dev, n});
    }
    return n > 0 ? std::min<int64_t>(n, PairCfg::MAX_PAIRS) : PairCfg::MAX_PAIRS;
}

// Schedule of the fused GEMM over its T tiles (S k-steps each) on P resident
// pairs: data-parallel when the tiles fill the pairs' rounds well enough
// (at most one round, a whole number of rounds, or a last round at least half
// full); stream-K over every tile when there are fewer tiles than half the
// pairs (on at most three pairs per tile: each more partial to add back
// costs the finishing pair more than the shorter share saves); otherwise
// whole data-parallel rounds with the last one-and-a-fraction rounds
// stream-K. When the activation operand is larger than three quarters of
// the L2 (big_act), the stream-K phase covers only the R = T mod P tiles left if
// every pair's share of them is at least a third of a tile (so at most four
// pairs share a tile): its pairs work at unrelated k offsets and share no
// activation reads through L2, and with a 235 MB activation (4096 x 28672) a
// stream-K phase over P + R tiles read about ten times the activation bytes
// from DRAM. With an activation that stays in L2 the longer phase is
// slightly faster (fewer, longer shares).
struct GemmSched {
    int64_t dp_tiles, pairs;
};
GemmSched gemm_sched(int64_t T, int64_t S, int64_t P, bool big_act) {
    if (2 * T < P) return {0, std::min({P, T * S, 3 * T})};
    if (T <= P || T % P == 0 || 2 * (T % P) >= P) return {T, std::min(P, T)};
    if (big_act && (T % P) * S / P >= (S + 2) / 3) return {(T / P) * P, P};
    return {(T / P - 1) * P, P};
}

// Activation bytes of one band of row tiles at most (gemm_pair.cuh, tile
// order): measured on the 70B-shaped layer, bands of 4 row tiles (32 MB) for
// an 8192-deep contraction and of 1-2 for a 28672-deep one were fastest; bands
// of 8 re-read a 64 MB activation from DRAM every data-parallel round.
constexpr int64_t kBandBytes = 32ll << 20;

// Activation operand size above which the stream-K phase is kept short:
// three quarters of the B300's 126 MB L2.
constexpr int64_t kBigActBytes = 96ll << 20;

// Sets prm.tile_rows and prm.dp_tiles for P resident pairs; returns the pairs
// to launch. Very few tiles of 512 rows (fewer than a quarter of the pairs):
// tiles of 256 rows instead, twice as many for the pairs to share (the
// decoded weight tile then feeds only 256 rows per k-step, so this pays only
// when the pairs would otherwise sit mostly idle).
int64_t gemm_schedule(TcParams &prm, int64_t P) {
    const int64_t nt = cdiv(prm.Nd, PairCfg::BN);
    prm.tile_rows = 4 * nt * cdiv(prm.M, PairCfg::PAIR_M) < P ? PairCfg::PAIR_M / 2 : PairCfg::PAIR_M;
    const bool big_act = prm.M * prm.nk_main * kGemmBK * 2 > kBigActBytes;
    const int64_t row_tile_bytes = (int64_t)prm.tile_rows * prm.nk_main * kGemmBK * 2;
    prm.band = 8;
    while (prm.band > 1 && prm.band * row_tile_bytes > kBandBytes) prm.band /= 2;
    const GemmSched sc =
        gemm_sched(nt * cdiv(prm.M, (int64_t)prm.tile_rows), prm.nk_main + prm.lora_steps, P, big_act);
    prm.dp_tiles = sc.dp_tiles;
    return sc.pairs;
}

// Launches the fused GEMM (forward or dX): a persistent grid of CTA pairs (no
// more than the device holds at once) on the schedule above, launched as a
// programmatic dependent of the preceding kernel.
template <int MODE>
qlora_status launch_gemm(GemmMaps &tm, TcParams prm, cudaStream_t s) {
    // output tiles leave through a tensor map (32 x 64 boxes, 128-byte
    // swizzle) when its row pitch and base allow one
    for (int g = 0; g < prm.ncg; ++g) {
        TcProj &o = prm.pj[g];
        o.out_v4 = (reinterpret_cast<uintptr_t>(o.out) & 15) == 0 && (o.ldo & 7) == 0;
        if (o.out_v4) {
            const qlora_status st = make_map(&tm.out[g], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, o.out, o.ncols, prm.M,
                                             o.ldo * 2, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B, "output");
            if (st) return st;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    const int64_t pairs = gemm_schedule(prm, gemm_pairs_resident<MODE>());
    cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
    cfg.blockDim = dim3(PairCfg::THREADS);
    cfg.dynamicSmemBytes = PairCfg::SMEM_BYTES;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cfg.stream = s;
    cudaError_t e;
    {
        ProfScope ps(MODE == kFwd ? QLORA_KERNEL_FWD_GEMM : QLORA_KERNEL_DX_GEMM, s);
        e = cudaLaunchKernelEx(&cfg, k_gemm_pair<MODE>, tm, prm);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(QLORA_ERR_CUDA, "fused GEMM launch failed: %s", cudaGetErrorString(e));
    }
    return launch_check("fused GEMM");
}

constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s per bounded wait
uint64_t wait_ns() { return g_wait_limit > 0 ? (uint64_t)g_wait_limit * 1000ull : kDefaultWaitNs; }

// One skinny problem: its operand maps, split plan and output.
struct SkJob {
    const CUtensorMap *ta, *tb;
    SkPlan pl;
    int mode;
    float scale;
    uint16_t *o16a;
    int lda;
    uint16_t *o16b;
    int ldb;
    float *o32;
    int zend = -1;  // zero columns [r, zend) of o16b (-1: up to ldb)
};

SkParams sk_params(const SkJob &j, int r, unsigned id) {
    SkParams prm{};
    prm.rows = j.pl.rows;
    prm.L = j.pl.L;
    prm.steps_per_chunk = j.pl.spc;
    prm.nchunks = (int)j.pl.chunks;
    prm.r = r;
    prm.s = j.scale;
    prm.mode = j.mode;
    prm.o16a = j.o16a;
    prm.lda = j.lda;
    prm.o16b = j.o16b;
    prm.ldb = j.ldb;
    prm.zend = j.zend < 0 ? j.ldb : j.zend;
    prm.o32 = j.o32;
    prm.wait_ns = wait_ns();
    prm.kernel_id = id;
    return prm;
}

// Largest number of clusters of `c` CTAs of this kernel that the device
// holds at once (cached per cluster size; 0 if the query fails).
template <int A_MN, int B_MN>
int skinny_max_clusters(int c) {
    static std::mutex mu;
    static std::vector<std::pair<int, std::array<int, 9>>> caches;  // per device
    const int dev = current_device();
    std::lock_guard<std::mutex> g(mu);
    std::array<int, 9> *cachep = nullptr;
    for (auto &d : caches)
        if (d.first == dev) cachep = &d.second;
    if (!cachep) {
        caches.push_back({dev, {-1, -1, -1, -1, -1, -1, -1, -1, -1}});
        cachep = &caches.back().second;
    }
    std::array<int, 9> &cache = *cachep;
    if (cache[c] < 0) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, (unsigned)c, 1);
        cfg.blockDim = dim3(SkCfg::THREADS);
        cfg.dynamicSmemBytes = SkCfg::SMEM_BYTES;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = (unsigned)c;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, k_lora_skinny<A_MN, B_MN>, &cfg) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        cache[c] = n;
    }
    return cache[c];
}

// Contraction chunks per tile: the largest cluster size (at most 8, and at
// least 4 steps of 64 per chunk) for which every tile's cluster is resident
// at once, so the launch runs as a single wave.
template <int A_MN, int B_MN>
int64_t skinny_chunks(int64_t clusters, int64_t steps) {
    for (int64_t c = std::min<int64_t>(8, steps / 4); c > 1; --c)
        if (skinny_max_clusters<A_MN, B_MN>((int)c) >= clusters) return c;
    return 1;
}

// Launches up to kSkMaxJobs skinny problems of one kind and rank-tile count
// (rs[j]: problem j's rank) in one grid; the first launch's problem 0 zeroes
// `zero` (the stream-K flags of the GEMM that follows).
template <int A_MN, int B_MN>
qlora_status run_skinny_jobs(const SkJob *jobs, const int *rs, int n, cudaStream_t s, unsigned id,
                             uint32_t *zero = nullptr, int nzero = 0) {
    if (n < 1 || n > kSkMaxJobs) return fail(QLORA_ERR_CUDA, "internal: %d skinny problems in one launch", n);
    const cudaError_t err = smem_attr(k_lora_skinny<A_MN, B_MN>, SkCfg::SMEM_BYTES);
    if (err != cudaSuccess) return fail(QLORA_ERR_CUDA, "setting shared memory size: %s", cudaGetErrorString(err));
    int64_t tiles = 0, max_steps = 1;
    for (int j = 0; j < n; ++j) {
        if (jobs[j].pl.zt != jobs[0].pl.zt)
            return fail(QLORA_ERR_CUDA, "internal: batched skinny problems differ in rank tiles");
        tiles += jobs[j].pl.tiles;
        max_steps = std::max<int64_t>(max_steps, cdiv(jobs[j].pl.L, 64));
    }
    const int64_t chunks = skinny_chunks<A_MN, B_MN>(tiles * jobs[0].pl.zt, max_steps);
    SkMaps tm;
    memset(&tm, 0, sizeof tm);
    SkBatch bt;
    memset(&bt, 0, sizeof bt);
    bt.n = n;
    for (int j = 0; j < n; ++j) {
        SkJob jb = jobs[j];
        jb.pl.spc = std::max<int64_t>(1, cdiv(std::max<int64_t>(1, cdiv(jb.pl.L, 64)), chunks));
        jb.pl.chunks = chunks;
        tm.a[j] = *jb.ta;
        tm.b[j] = *jb.tb;
        bt.p[j] = sk_params(jb, rs[j], id);
        bt.first[j + 1] = bt.first[j] + (int)jb.pl.tiles;
    }
    bt.p[0].zero = zero;
    bt.p[0].nzero = nzero;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)tiles, (unsigned)chunks, (unsigned)jobs[0].pl.zt);
    cfg.blockDim = dim3(SkCfg::THREADS);
    cfg.dynamicSmemBytes = SkCfg::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = (unsigned)chunks;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = chunks > 1 ? 2 : 1;
    cudaError_t e;
    {
        ProfScope ps(jobs[0].mode >= kRedDA ? QLORA_KERNEL_GRADS : QLORA_KERNEL_LORA_PRE, s);
        e = cudaLaunchKernelEx(&cfg, k_lora_skinny<A_MN, B_MN>, tm, bt);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(QLORA_ERR_CUDA, "k_lora_skinny: launch failed: %s", cudaGetErrorString(e));
    }
    return launch_check("k_lora_skinny");
}

// One skinny problem, or two (j1 != null) of the same kind and rank.
template <int A_MN, int B_MN>
qlora_status run_skinny(SkJob j0, const SkJob *j1p, int r, cudaStream_t s, unsigned id, uint32_t *zero = nullptr,
                        int nzero = 0) {
    const SkJob jobs[2] = {j0, j1p ? *j1p : j0};
    const int rs[2] = {r, r};
    return run_skinny_jobs<A_MN, B_MN>(jobs, rs, j1p ? 2 : 1, s, id, zero, nzero);
}

}  // namespace

// One few-token forward launch pair with parameters for NP projections.
template <int NP, class Kern>
static qlora_status few_fwd_launch_np(Kern kern, const uint16_t *X16, int64_t M, const Wt *const *w,
                                      const void *const *A, const void *const *B, void *const *Y, int n, int r,
                                      float scale, uint16_t *U16, int ldu, uint16_t *sU, int rp, float *slots,
                                      uint32_t *counters, cudaStream_t s) {
    qlora_status st;
    const int64_t K = w[0]->cols;
    const cudaError_t aerr = smem_attr(kern, FewCfg::SMEM_BYTES);
    if (aerr != cudaSuccess) return fail(QLORA_ERR_CUDA, "setting shared memory size: %s", cudaGetErrorString(aerr));
    FewParams<NP> prm{};
    FewMaps<NP> maps;
    memset(&maps, 0, sizeof maps);
    const uint16_t *da[kMaxGroup] = {nullptr, nullptr, nullptr, nullptr};
    int64_t tiles = 0;
    // code boxes of 128 bytes x 32 rows (FewCfg::TASK_BYTES, one task),
    // 128-byte swizzle
    static_assert(FewCfg::TASK_BYTES == 128 * FewCfg::ROWS, "code box");
    for (int g = 0; g < n; ++g) {
        const Wt &wg = *w[g];
        if ((st = make_map(&maps.codes[g], CU_TENSOR_MAP_DATA_TYPE_UINT8, wg.codes, K / 2, wg.rows, K / 2, 128,
                           FewCfg::ROWS, CU_TENSOR_MAP_SWIZZLE_128B, "codes")))
            return st;
        FewProj &pr = prm.proj[g];
        pr.q = wg.q;
        pr.s2 = wg.s2;
        pr.mean = wg.mean;
        pr.absmax = wg.absmax;
        pr.B = static_cast<const uint16_t *>(B[g]);
        pr.Y = static_cast<uint16_t *>(Y[g]);
        pr.N = wg.rows;
        pr.tile0 = (uint32_t)tiles;
        pr.sucol = g * rp;
        tiles += cdiv(wg.rows, FewCfg::ROWS);
        da[g] = static_cast<const uint16_t *>(A[g]);
    }
    const FewPlan fp = few_plan_tiles(M, tiles, K);
    {
        // a programmatic dependent of the preceding kernel (it waits for
        // that grid before touching memory): its launch overlaps the
        // preceding kernel's end
        cudaLaunchConfig_t dc = {};
        dc.gridDim = dim3((unsigned)M, (unsigned)r, (unsigned)n);
        dc.blockDim = dim3(kFewDownThreads);
        dc.stream = s;
        cudaLaunchAttribute dattr[1];
        dattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        dattr[0].val.programmaticStreamSerializationAllowed = 1;
        dc.attrs = dattr;
        dc.numAttrs = 1;
        ProfScope ps(QLORA_KERNEL_LORA_PRE, s);
        const cudaError_t de = cudaLaunchKernelEx(&dc, k_few_down, X16, (int64_t)K, da[0], da[1], da[2], da[3], r,
                                                  scale, U16, ldu, sU, n * rp, rp, counters, (int)tiles);
        if (de != cudaSuccess) {
            cudaGetLastError();
            return fail(QLORA_ERR_CUDA, "k_few_down: launch failed: %s", cudaGetErrorString(de));
        }
    }
    if ((st = launch_check("k_few_down"))) return st;
    prm.X = X16;
    prm.M = M;
    prm.K = K;
    prm.sU = sU;
    prm.ldu = n * rp;
    prm.r = r;
    prm.nproj = n;
    prm.slots = slots;
    prm.counters = counters;
    prm.tasks = fp.tasks;
    prm.tpr = fp.tpr;
    prm.warps = fp.warps;
    prm.wait_ns = wait_ns();
    {
        static const float kLevels[2][16] = {QLORA_NF4_LEVELS, QLORA_INT4_LEVELS};
        memcpy(prm.levels, kLevels[w[0]->tab], sizeof prm.levels);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)fp.grid);
    cfg.blockDim = dim3((unsigned)(32 * fp.wpc));
    cfg.dynamicSmemBytes = FewCfg::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    {
        ProfScope ps(QLORA_KERNEL_FWD_SIMT, s);
        e = cudaLaunchKernelEx(&cfg, kern, maps, prm);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(QLORA_ERR_CUDA, "k_fwd_few: launch failed: %s", cudaGetErrorString(e));
    }
    return launch_check("k_fwd_few");
}

extern "C" {

const char *qlora_version(void) { return "qlora-b300 0.1 (sm_103a)"; }

int64_t qlora_debug_few_split(int64_t M, int64_t N, int64_t K, int64_t *out, int64_t cap) {
    if (M < 1 || M > 8 * FewCfg::MAX_NT || N < 1 || K < FewCfg::TK || K % FewCfg::TK || !out ||
        N * (K / kBlock) >= (int64_t(1) << 31))
        return -2;
    const FewPlan f = few_plan(M, N, K);
    const int64_t need = 4 + 2 * f.warps + 2 * f.tiles;
    if (cap < need) return -1;
    const uint32_t T = (uint32_t)f.tasks, W = (uint32_t)f.warps, P = (uint32_t)f.tpr;
    out[0] = f.tasks;
    out[1] = f.warps;
    out[2] = f.tpr;
    out[3] = f.tiles;
    for (uint32_t w = 0; w < W; ++w) {
        out[4 + 2 * w] = few_begin(w, W, T);
        out[5 + 2 * w] = few_begin(w + 1, W, T);
    }
    for (int64_t t = 0; t < f.tiles; ++t) {
        out[4 + 2 * f.warps + 2 * t] = few_owner((uint32_t)t * P, W, T);
        out[5 + 2 * f.warps + 2 * t] = few_owner((uint32_t)(t + 1) * P - 1, W, T);
    }
    return need;
}

int64_t qlora_debug_gemm_segments(int64_t M, int64_t Nd, int64_t nk_main, int lora_steps, int pairs_resident,
                                  int64_t *out, int64_t cap) {
    if (M < 1 || Nd < 1 || nk_main < 0 || lora_steps < 0 || nk_main + lora_steps < 1 || pairs_resident < 1 ||
        pairs_resident > PairCfg::MAX_PAIRS || !out)
        return -2;
    if (cap < 4) return -1;
    TcParams prm{};
    prm.M = M;
    prm.Nd = Nd;
    prm.nk_main = nk_main;
    prm.lora_steps = lora_steps;
    prm.ncg = prm.nkg = 1;
    prm.cg_first[1] = cdiv(Nd, PairCfg::BN);
    prm.kg_first[1] = nk_main;
    const int64_t pairs = gemm_schedule(prm, pairs_resident);
    const PairPlan pl = make_plan(prm, pairs);
    out[0] = prm.tile_rows;
    out[1] = prm.dp_tiles;
    out[2] = pairs;
    out[3] = pl.T;
    int64_t n = 4;
    for (int64_t q = 0; q < pairs; ++q) {
        SegWalk sw = seg_walk(pl, q);
        PairSeg w;
        while (seg_next(prm, pl, sw, w)) {
            if (n + 9 > cap) return -1;
            // the same head / contributor computation as the kernel's epilogue
            const int64_t h = w.role == kSegPart ? head_pair(pl, q, w.t) : q;
            out[n++] = q;
            out[n++] = w.t;
            out[n++] = w.m0;
            out[n++] = w.c0;
            out[n++] = w.kbeg;
            out[n++] = w.nk;
            out[n++] = w.role;
            out[n++] = h;
            out[n++] = w.role == kSegFull ? 1 : head_contrib_end(pl, h, w.t) - h;
        }
    }
    return (n - 4) / 9;
}

#ifdef QLORA_GEMM_STAMPS
// Diagnostic build only (not part of the ABI header): copies the fused GEMM's
// timeline of the last launch (8 rows of kStampSteps globaltimer values, row
// meanings in gemm_pair.cuh) to `host`; 0 on success.
int qlora_debug_gemm_stamps(unsigned long long *host) {
    return cudaMemcpyFromSymbol(host, d_gemm_stamps, sizeof(d_gemm_stamps)) == cudaSuccess ? 0 : 1;
}
// The few-token forward's per-warp timeline of the last launch
// (kFewStampWarps x 16 values, columns in fwd_few.cuh); 0 on success.
int qlora_debug_few_stamps(unsigned long long *host) {
    return cudaMemcpyFromSymbol(host, d_few_stamps, sizeof(d_few_stamps)) == cudaSuccess ? 0 : 1;
}
#endif

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

static qlora_status quantize_impl(const void *W, const Wt &out, void *ws, size_t ws_bytes, qlora_stream_t stream) {
    qlora_status st = check_weight(out, false);
    if (st) return st;
    if (!W) return fail(QLORA_ERR_NULL, "W is NULL");
    if (!al16(W)) return fail(QLORA_ERR_ALIGN, "W must be 16-byte aligned");
    const int64_t rows = out.rows, cols = out.cols;
    if (rows == 0) return ok();
    if (out.absmax) {
        if ((st = quantize_launch(W, out, nullptr, nullptr, nullptr, nullptr, reinterpret_cast<cudaStream_t>(stream))))
            return st;
        return ok();
    }
    if (!ws) return fail(QLORA_ERR_NULL, "workspace is NULL");
    if (!al16(ws)) return fail(QLORA_ERR_ALIGN, "workspace must be 16-byte aligned");
    float *absmax;
    double *gsum, *b0, *b1;
    const size_t need = quantize_ws(rows, cols, &absmax, &gsum, &b0, &b1, ws);
    if (ws_bytes < need)
        return fail(QLORA_ERR_WORKSPACE, "quantize workspace %zu < %zu bytes", ws_bytes, need);
    return quantize_launch(W, out, absmax, gsum, b0, b1, reinterpret_cast<cudaStream_t>(stream));
}

qlora_status qlora_nf4_quantize(const void *W, qlora_nf4_weight *out, void *ws, size_t ws_bytes,
                                qlora_stream_t stream) {
    if (!out) return fail(QLORA_ERR_NULL, "weight descriptor is NULL");
    return quantize_impl(W, wt_of(out), ws, ws_bytes, stream);
}

qlora_status qlora_q4_quantize(const void *W, qlora_q4_weight *out, void *ws, size_t ws_bytes, qlora_stream_t stream) {
    if (!out) return fail(QLORA_ERR_NULL, "weight descriptor is NULL");
    return quantize_impl(W, wt_of(out), ws, ws_bytes, stream);
}

// ---- quantize without a caller workspace ------------------------------------
// The scratch lives in this file-scope device array. In host code its name is
// only a host-side stand-in, so its device address is looked up with
// cudaGetSymbolAddress. A __device__ array has one instance per CUDA context,
// so the address is cached per context (the current one at the call), which
// covers a host that drives the same GPU through several contexts.
static __device__ __align__(256) unsigned char g_quantize_scratch[QLORA_NF4_NOALLOC_SCRATCH_BYTES];
static std::mutex g_scratch_mu;
static std::vector<std::pair<CUcontext, void *>> g_scratch_ptr;

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);

static CtxGetCurrentFn ctx_get_current_fn() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(f);
    });
    return fn;
}

static qlora_status quantize_scratch(void **out) {
    CtxGetCurrentFn get = ctx_get_current_fn();
    if (!get) return fail(QLORA_ERR_UNSUPPORTED, "cuCtxGetCurrent is not available from the driver");
    CUcontext ctx = nullptr;
    if (get(&ctx) != CUDA_SUCCESS) return fail(QLORA_ERR_CUDA, "cannot read the current CUDA context");
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (ctx) {
        for (const auto &c : g_scratch_ptr)
            if (c.first == ctx) {
                *out = c.second;
                return QLORA_OK;
            }
    }
    // first call in this context (with no context current yet, the runtime
    // binds the current device's primary context here)
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_quantize_scratch);
    if (e != cudaSuccess || !p) return fail(QLORA_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    if (!ctx && (get(&ctx) != CUDA_SUCCESS || !ctx)) return fail(QLORA_ERR_CUDA, "no current CUDA context");
    g_scratch_ptr.push_back({ctx, p});
    *out = p;
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
    return quantize_launch(W, wt_of(out), absmax, gsum, b0, b1, reinterpret_cast<cudaStream_t>(stream));
}

size_t qlora_lora_merge_workspace(int64_t rows, int64_t cols) {
    if (!valid_dims(rows, cols) || rows == 0) return 0;
    return up((size_t)(rows * cols) * 2, 256) + quantize_ws(rows, cols, nullptr, nullptr, nullptr, nullptr, nullptr);
}

qlora_status qlora_lora_merge_requantize(const qlora_nf4_weight *w, const void *A, const void *B, int r, float scale,
                                         qlora_nf4_weight *out, void *ws, size_t ws_bytes, qlora_stream_t stream) {
    qlora_status st = check_weight(w, false);
    if (st) return st;
    if ((st = check_weight(out, false))) return st;
    if (out->rows != w->rows || out->cols != w->cols)
        return fail(QLORA_ERR_SHAPE, "merged weight [%lld, %lld] differs from the base [%lld, %lld]",
                    (long long)out->rows, (long long)out->cols, (long long)w->rows, (long long)w->cols);
    if (r < 1 || r > 128) return fail(QLORA_ERR_RANK, "LoRA rank r = %d outside [1, 128]", r);
    if (!A || !B) return fail(QLORA_ERR_NULL, "LoRA A or B is NULL");
    if (!al16(A) || !al16(B)) return fail(QLORA_ERR_ALIGN, "LoRA A and B must be 16-byte aligned");
    const int64_t N = w->rows, K = w->cols;
    if (N == 0) return ok();
    if (!ws) return fail(QLORA_ERR_NULL, "workspace is NULL");
    if (!al16(ws)) return fail(QLORA_ERR_ALIGN, "workspace must be 16-byte aligned");
    const size_t need = qlora_lora_merge_workspace(N, K);
    if (ws_bytes < need) return fail(QLORA_ERR_WORKSPACE, "merge workspace %zu < %zu bytes", ws_bytes, need);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint16_t *merged = static_cast<uint16_t *>(ws);
    const int64_t chunks = N * K / 8;
    {
        ProfScope ps(QLORA_KERNEL_QUANTIZE, s);
        k_lora_merge<<<(unsigned)cdiv(chunks, 256), 256, 0, s>>>(
            reinterpret_cast<const uint32_t *>(w->codes), w->absmax_q, w->absmax_scale, w->absmax_mean, N, K,
            static_cast<const uint16_t *>(A), static_cast<const uint16_t *>(B), r, scale,
            reinterpret_cast<uint4 *>(merged));
    }
    if ((st = launch_check("k_lora_merge"))) return st;
    float *absmax;
    double *gsum, *b0, *b1;
    quantize_ws(N, K, &absmax, &gsum, &b0, &b1, static_cast<char *>(ws) + up((size_t)(N * K) * 2, 256));
    return quantize_launch(merged, wt_of(out), absmax, gsum, b0, b1, s);
}

// A pointer the device can dereference: device or managed memory, or host
// memory that is pinned (registered); pageable host memory is not.
static bool device_reachable(const void *ptr) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged ||
           (a.type == cudaMemoryTypeHost && a.devicePointer == ptr);
}

qlora_status qlora_adamw_step(float *param, uint16_t *param_bf16, const float *grad, float *m, float *v, int64_t n,
                              float lr, float beta1, float beta2, float eps, float weight_decay, int64_t step,
                              qlora_stream_t stream) {
    if (n < 0) return fail(QLORA_ERR_SHAPE, "n = %lld < 0", (long long)n);
    if (step < 1) return fail(QLORA_ERR_SHAPE, "step = %lld < 1", (long long)step);
    if (n == 0) return ok();
    if (!param || !grad || !m || !v) return fail(QLORA_ERR_NULL, "param, grad, m or v is NULL");
    if (!al16(param) || !al16(grad) || !al16(m) || !al16(v) || (param_bf16 && (reinterpret_cast<uintptr_t>(param_bf16) & 7)))
        return fail(QLORA_ERR_ALIGN, "param, grad, m, v must be 16-byte aligned, param_bf16 8-byte aligned");
    if (!(beta1 >= 0.0f && beta1 < 1.0f && beta2 >= 0.0f && beta2 < 1.0f && eps > 0.0f))
        return fail(QLORA_ERR_SHAPE, "need 0 <= beta1, beta2 < 1 and eps > 0");
    const void *ptrs[5] = {param, grad, m, v, param_bf16};
    for (int i = 0; i < 5; ++i)
        if (ptrs[i] && !device_reachable(ptrs[i]))
            return fail(QLORA_ERR_UNSUPPORTED, "pointer %d is not reachable from the device (pageable host memory?)", i);
    AdamwParams h;
    const double b1t = 1.0 - pow((double)beta1, (double)step), b2t = 1.0 - pow((double)beta2, (double)step);
    h.decay = (float)(1.0 - (double)lr * (double)weight_decay);
    h.b1 = beta1;
    h.b2 = beta2;
    h.one_m_b1 = 1.0f - beta1;
    h.one_m_b2 = 1.0f - beta2;
    h.step = (float)((double)lr / b1t);
    h.c2 = (float)sqrt(b2t);
    h.eps = eps;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const unsigned grid = (unsigned)std::min<int64_t>(std::max<int64_t>(1, cdiv(n / 4, 256)), 148 * 8);
    {
        ProfScope ps(QLORA_KERNEL_OPTIM, s);
        k_adamw<<<grid, 256, 0, s>>>(param, param_bf16, grad, m, v, n, h);
    }
    qlora_status st = launch_check("k_adamw");
    if (st) return st;
    return ok();
}

static qlora_status dequantize_impl(const Wt &w, void *out, qlora_stream_t stream) {
    qlora_status st = check_weight(w, false);
    if (st) return st;
    if (!out) return fail(QLORA_ERR_NULL, "output is NULL");
    if (!al16(out)) return fail(QLORA_ERR_ALIGN, "output must be 16-byte aligned");
    if (w.rows == 0) return ok();
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t nb = w.rows * w.cols / kBlock;
    const cudaError_t aerr = smem_attr(k_nf4_dequant, kDeqSmem);
    if (aerr != cudaSuccess) return fail(QLORA_ERR_CUDA, "setting shared memory size: %s", cudaGetErrorString(aerr));
    // the output viewed as [blocks, 64] bf16 rows of 128 bytes
    CUtensorMap tmO;
    if ((st = make_map(&tmO, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, out, kBlock, nb, kBlock * 2, 64, 32,
                       CU_TENSOR_MAP_SWIZZLE_128B, "output")))
        return st;
    const int64_t nchunks = cdiv(nb, 32);
    const unsigned grid = (unsigned)std::min<int64_t>(cdiv(nchunks, kDeqWarps), 148 * 3);
    {
        ProfScope ps(QLORA_KERNEL_DEQUANT, s);
        k_nf4_dequant<<<grid, kDeqWarps * 32, kDeqSmem, s>>>(tmO, reinterpret_cast<const uint4 *>(w.codes), w.q,
                                                             w.s2, w.mean, nb, w.absmax, w.tab);
    }
    if ((st = launch_check("k_nf4_dequant"))) return st;
    return ok();
}

qlora_status qlora_nf4_dequantize(const qlora_nf4_weight *w, void *out, qlora_stream_t stream) {
    if (!w) return fail(QLORA_ERR_NULL, "weight descriptor is NULL");
    return dequantize_impl(wt_of(w), out, stream);
}

qlora_status qlora_q4_dequantize(const qlora_q4_weight *w, void *out, qlora_stream_t stream) {
    if (!w) return fail(QLORA_ERR_NULL, "weight descriptor is NULL");
    return dequantize_impl(wt_of(w), out, stream);
}

size_t qlora_linear_fwd_workspace(int64_t M, const qlora_nf4_weight *w, int r) {
    if (!w || !valid_dims(w->rows, w->cols) || M < 0 || r < 1 || r > 128) return 0;
    return fwd_ws(M, w->rows, w->cols, r, nullptr, nullptr);
}

size_t qlora_linear_bwd_workspace(int64_t M, const qlora_nf4_weight *w, int r) {
    if (!w || !valid_dims(w->rows, w->cols) || M < 0 || r < 1 || r > 128) return 0;
    return bwd_ws(M, w->rows, w->cols, r, nullptr, nullptr);
}

size_t qlora_q4_linear_fwd_workspace(int64_t M, const qlora_q4_weight *w, int r) {
    if (!w || !valid_dims(w->rows, w->cols) || M < 0 || r < 1 || r > 128) return 0;
    return fwd_ws(M, w->rows, w->cols, r, nullptr, nullptr);
}

size_t qlora_q4_linear_bwd_workspace(int64_t M, const qlora_q4_weight *w, int r) {
    if (!w || !valid_dims(w->rows, w->cols) || M < 0 || r < 1 || r > 128) return 0;
    return bwd_ws(M, w->rows, w->cols, r, nullptr, nullptr);
}

static qlora_status check_linear_common(int64_t M, const Wt &w, const void *A, const void *B, int r, void *ws) {
    qlora_status st = check_weight(w, true);
    if (st) return st;
    if (M < 0 || M >= kMaxDim) return fail(QLORA_ERR_SHAPE, "M = %lld out of range", (long long)M);
    if (r < 1 || r > 128) return fail(QLORA_ERR_RANK, "LoRA rank r = %d outside [1, 128]", r);
    if (!A || !B) return fail(QLORA_ERR_NULL, "LoRA A or B is NULL");
    if (!al16(A) || !al16(B)) return fail(QLORA_ERR_ALIGN, "LoRA A and B must be 16-byte aligned");
    if (ws && !al16(ws)) return fail(QLORA_ERR_ALIGN, "workspace must be 16-byte aligned");
    return QLORA_OK;
}

// The few-token forward of n projections (1..kMaxGroup) sharing X and K:
// k_few_down (sU of all of them, slices of rp columns, lds = n rp) then one
// k_fwd_few over the row tiles of all of them. Workspace: sU [M, n rp],
// slots (few_slot_floats(M) per warp of the plan), one counter per row tile.
static qlora_status few_fwd_launch(const uint16_t *X16, int64_t M, const Wt *const *w, const void *const *A,
                                   const void *const *B, void *const *Y, int n, int r, float scale, uint16_t *U16,
                                   int ldu, uint16_t *sU, int rp, float *slots, uint32_t *counters, cudaStream_t s) {
    qlora_status st;
    if ((st = tc_device_ok())) return st;
    if (n > 1)  // several projections: NF4 with double quantization only (the group calls)
        return few_fwd_launch_np<kMaxGroup>(M <= 8 ? k_fwd_few<1, false, true> : k_fwd_few<2, false, true>, X16, M,
                                            w, A, B, Y, n, r, scale, U16, ldu, sU, rp, slots, counters, s);
    const bool f32a = w[0]->absmax != nullptr;
    auto kern = M <= 8 ? (f32a ? k_fwd_few<1, true, false> : k_fwd_few<1, false, false>)
                       : (f32a ? k_fwd_few<2, true, false> : k_fwd_few<2, false, false>);
    return few_fwd_launch_np<1>(kern, X16, M, w, A, B, Y, n, r, scale, U16, ldu, sU, rp, slots, counters, s);
}

// ldu: row pitch (elements) of U_save; r for the single-layer entry points.
static qlora_status linear_fwd_impl(const void *X, int64_t M, const Wt &w, const void *A, const void *B, int r,
                                    float scale, void *Y, void *U_save, void *ws, size_t ws_bytes,
                                    qlora_stream_t stream, int ldu) {
    qlora_status st = check_linear_common(M, w, A, B, r, ws);
    if (st) return st;
    if (M > 0 && (!X || !Y)) return fail(QLORA_ERR_NULL, "X or Y is NULL");
    if ((X && !al16(X)) || (Y && !al16(Y)) || (U_save && !al16(U_save)))
        return fail(QLORA_ERR_ALIGN, "X, Y and U_save must be 16-byte aligned");
    if (M == 0) return ok();
    const int64_t N = w.rows, K = w.cols;
    FwdWs f;
    const size_t need = fwd_ws(M, N, K, r, ws, &f);
    if (!ws) return fail(QLORA_ERR_NULL, "workspace is NULL");
    if (ws_bytes < need) return fail(QLORA_ERR_WORKSPACE, "forward workspace %zu < %zu bytes", ws_bytes, need);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int rp = lora_pad(r);
    const uint16_t *X16 = static_cast<const uint16_t *>(X);
    uint16_t *U16 = static_cast<uint16_t *>(U_save);

    if (few_path(M, N, K)) {
        // few tokens, K a multiple of 256: persistent HBM-bound kernel
        const Wt *wp = &w;
        return few_fwd_launch(X16, M, &wp, &A, &B, &Y, 1, r, scale, U16, ldu, f.sU, rp, f.few_slots, f.few_counters,
                              s);
    }

    if (M <= kSmallMaxM && K <= kSmallMaxK) {
        // few tokens: HBM-bound path (mma.sync over the decoded weight rows)
        if ((st = tc_device_ok())) return st;
        {
            ProfScope ps(QLORA_KERNEL_LORA_PRE, s);
            k_lora_down<<<(unsigned)(M * rp), kDownThreads, 0, s>>>(X16, M, K, static_cast<const uint16_t *>(A), r, scale,
                                                              U16, ldu, f.sU, rp);
        }
        if ((st = launch_check("k_lora_down"))) return st;
        CUtensorMap tmC;
        if ((st = make_map(&tmC, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.codes, K / 2, N, K / 2, 128, SmallCfg::ROWS,
                           CU_TENSOR_MAP_SWIZZLE_128B, "codes")))
            return st;
        const unsigned grid = (unsigned)cdiv(N, SmallCfg::ROWS);
        const int nt = M <= 8 ? 1 : (M <= 16 ? 2 : 4);
        {
            ProfScope ps(QLORA_KERNEL_FWD_SIMT, s);
            auto kern = nt == 1 ? k_fwd_small<1> : (nt == 2 ? k_fwd_small<2> : k_fwd_small<4>);
            // a programmatic dependent of k_lora_down: the weights stream
            // while U is computed
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(grid);
            cfg.blockDim = dim3(SmallCfg::THREADS);
            cfg.stream = s;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, tmC, (const uint16_t *)X16, M, K,
                                                     (const int8_t *)w.q, (const float *)w.s2, (const float *)w.mean,
                                                     N, (const uint16_t *)f.sU, rp, static_cast<const uint16_t *>(B),
                                                     r, static_cast<uint16_t *>(Y), wait_ns(),
                                                     (const float *)w.absmax, w.tab);
            if (e != cudaSuccess) {
                cudaGetLastError();
                return fail(QLORA_ERR_CUDA, "k_fwd_small: launch failed: %s", cudaGetErrorString(e));
            }
        }
        if ((st = launch_check("k_fwd_small"))) return st;
        return ok();
    }

    if ((st = tc_device_ok()) || (st = tc_setup<kFwd>())) return st;
    const int rs = lora_rs(r);
    // B as the LoRA tile of the GEMM: [N, r] directly when its rows are 16-byte
    // multiples, else a copy with rows of rs (zero columns beyond r)
    const void *Bl = B;
    if (r % 8) {
        {
            ProfScope ps(QLORA_KERNEL_LORA_PRE, s);
            k_pad_cols<<<(unsigned)cdiv(N * rs, 256), 256, 0, s>>>(static_cast<const uint16_t *>(B), N, r, rs, f.Bp);
        }
        if ((st = launch_check("k_pad_cols(B)"))) return st;
        Bl = f.Bp;
    }
    GemmMaps gm;
    memset(&gm, 0, sizeof gm);
    CUtensorMap &tmX = gm.act[0];
    CUtensorMap tmA;
    if ((st = make_map(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, K, M, K * 2, 64, 128,
                       CU_TENSOR_MAP_SWIZZLE_128B, "X")) ||
        (st = make_map(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A, K, r, K * 2, 64, 64,
                       CU_TENSOR_MAP_SWIZZLE_128B, "A")) ||
        (st = make_map(&gm.codes[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, w.codes, K / 2, N, K / 2, 32, 128,
                       CU_TENSOR_MAP_SWIZZLE_32B, "codes")) ||
        (st = make_map(&gm.lact, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, f.sU, rs, M, rs * 2, 64, 128,
                       CU_TENSOR_MAP_SWIZZLE_128B, "sU")) ||
        (st = make_map(&gm.lw[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Bl, rs, N, rs * 2, 64, 128,
                       CU_TENSOR_MAP_SWIZZLE_128B, "B")))
        return st;
    // U = X A^T on the tensor cores; U (bf16) to U_save, s*U (bf16) to the workspace
    const SkPlan pu = sk_plan(M, K, r);
    if ((st = run_skinny<0, 0>(SkJob{&tmX, &tmA, pu, kRedU, scale, U16, ldu, f.sU, rs, nullptr}, nullptr, r, s, 3,
                               f.sk.flags, kSkFlagWords)))
        return st;
    TcParams prm{};
    prm.M = M;
    prm.Nd = N;
    prm.w_cols = K;
    prm.nk_main = K / kGemmBK;
    prm.lora_steps = rp / 64;
    prm.r = r;
    prm.tab = w.tab;
    prm.ncg = prm.nkg = 1;
    prm.cg_first[1] = cdiv(N, PairCfg::BN);
    prm.kg_first[1] = prm.nk_main;
    prm.pj[0] = TcProj{w.q, w.s2, w.mean, w.absmax, N, static_cast<uint16_t *>(Y), N, N, 0, 0};
    prm.flags = f.sk.flags;
    prm.slots = f.sk.slots;
    prm.wait_ns = wait_ns();
    prm.kernel_id = 1;
    if ((st = launch_gemm<kFwd>(gm, prm, s))) return st;
    return ok();
}

// ldu: row pitch (elements) of U_saved; r for the single-layer entry points
// (any multiple of 8 when r % 8 == 0).
static qlora_status linear_bwd_impl(const void *dY, const void *X, const void *U_saved, int64_t M, const Wt &w,
                                    const void *A, const void *B, int r, float scale, void *dX, float *dA, float *dB,
                                    void *ws, size_t ws_bytes, qlora_stream_t stream, int ldu_saved) {
    qlora_status st = check_linear_common(M, w, A, B, r, ws);
    if (st) return st;
    if (!dA || !dB) return fail(QLORA_ERR_NULL, "dA or dB is NULL");
    if (M > 0 && (!dY || !X || !dX)) return fail(QLORA_ERR_NULL, "dY, X or dX is NULL");
    if ((dY && !al16(dY)) || (X && !al16(X)) || (dX && !al16(dX)) || !al16(dA) || !al16(dB) ||
        (U_saved && !al16(U_saved)))
        return fail(QLORA_ERR_ALIGN, "dY, X, U_saved, dX, dA and dB must be 16-byte aligned");
    const int64_t N = w.rows, K = w.cols;
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
            k_lora_down<<<(unsigned)(M * rp), kDownThreads, 0, s>>>(dY16, M, N, b.Bt, r, scale, nullptr, 0, b.sV, rp);
        }
        if ((st = launch_check("k_lora_down(V)"))) return st;
        const uint16_t *U = static_cast<const uint16_t *>(U_saved);
        int ldu = ldu_saved;
        if (!U) {
            {
                ProfScope ps(QLORA_KERNEL_LORA_PRE, s);
                k_lora_down<<<(unsigned)(M * rp), kDownThreads, 0, s>>>(X16, M, K, A16, r, 1.0f, nullptr, 0, b.U, rp);
            }
            if ((st = launch_check("k_lora_down(U)"))) return st;
            U = b.U;
            ldu = rp;
        }
        dim3 grid((unsigned)cdiv(K, kSt), (unsigned)cdiv(M, kSt));
        {
            ProfScope ps(QLORA_KERNEL_DX_SIMT, s);
            k_dx_simt<<<grid, 256, 0, s>>>(dY16, M, N, w.codes, w.q, w.s2, w.mean, K, b.sV, rp, A16, r,
                                           static_cast<uint16_t *>(dX), w.absmax, w.tab);
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
    const int rs = lora_rs(r);
    // B [N, r] and U [M, r] are read by TMA directly when their rows are
    // 16-byte multiples (r % 8 == 0), else from copies with rows of rs
    const void *Bl = B16, *Ul = U_saved;
    if (r % 8) {
        {
            ProfScope ps(QLORA_KERNEL_LORA_PRE, s);
            k_pad_cols<<<(unsigned)cdiv(N * rs, 256), 256, 0, s>>>(B16, N, r, rs, b.Bp);
        }
        if ((st = launch_check("k_pad_cols(B)"))) return st;
        Bl = b.Bp;
        if (U_saved) {
            {
                ProfScope ps(QLORA_KERNEL_LORA_PRE, s);
                k_pad_cols<<<(unsigned)cdiv(M * rs, 256), 256, 0, s>>>(static_cast<const uint16_t *>(U_saved), M,
                                                                      r, rs, b.U);
            }
            if ((st = launch_check("k_pad_cols(U)"))) return st;
            Ul = b.U;
        }
    }
    if (!U_saved) Ul = b.U;
    const int ldb_l = r % 8 ? rs : r;
    CUtensorMap tmD, tmDmn, tmXk, tmXmn, tmC, tmV, tmA, tmBp, tmUp, tmVmn;
    if ((st = make_map(&tmD, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dY, N, M, N * 2, 64, 128,
                       CU_TENSOR_MAP_SWIZZLE_128B, "dY")) ||
        (st = make_map(&tmDmn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dY, N, M, N * 2, 64, 64,
                       CU_TENSOR_MAP_SWIZZLE_128B, "dY (MN)")) ||
        (st = make_map(&tmXk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, K, M, K * 2, 64, 128,
                       CU_TENSOR_MAP_SWIZZLE_128B, "X")) ||
        (st = make_map(&tmXmn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, K, M, K * 2, 64, 64,
                       CU_TENSOR_MAP_SWIZZLE_128B, "X (MN)")) ||
        (st = make_map(&tmC, CU_TENSOR_MAP_DATA_TYPE_UINT8, w.codes, K / 2, N, K / 2, 64, 64,
                       CU_TENSOR_MAP_SWIZZLE_64B, "codes")) ||
        (st = make_map(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, b.sV, rs, M, rs * 2, 64, 128,
                       CU_TENSOR_MAP_SWIZZLE_128B, "sV")) ||
        (st = make_map(&tmVmn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, b.sV, rs, M, rs * 2, 64, 64,
                       CU_TENSOR_MAP_SWIZZLE_128B, "sV (MN)")) ||
        (st = make_map(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A16, K, r, K * 2, 64, 64,
                       CU_TENSOR_MAP_SWIZZLE_128B, "A")) ||
        (st = make_map(&tmBp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Bl, ldb_l, N, ldb_l * 2, 64, 64,
                       CU_TENSOR_MAP_SWIZZLE_128B, "B")) ||
        (st = make_map(&tmUp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Ul, U_saved ? ldb_l : rs, M,
                       (U_saved ? (r % 8 ? rs : ldu_saved) : rs) * 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B, "U")))
        return st;
    // V = dY B -> sV = bf16(s * V)
    const SkPlan pv = sk_plan(M, N, r);
    if ((st = run_skinny<0, 1>(SkJob{&tmD, &tmBp, pv, kRedV, scale, nullptr, 0, b.sV, rs, nullptr}, nullptr, r, s,
                               4, b.sk.flags, kSkFlagWords)))
        return st;
    // U recomputed as X A^T when the forward's U is not given
    if (!U_saved) {
        CUtensorMap tmAk;
        if ((st = make_map(&tmAk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, A16, K, r, K * 2, 64, 64,
                           CU_TENSOR_MAP_SWIZZLE_128B, "A")))
            return st;
        const SkPlan pu = sk_plan(M, K, r);
        if ((st = run_skinny<0, 0>(SkJob{&tmXk, &tmAk, pu, kRedV, 1.0f, nullptr, 0, b.U, rs, nullptr}, nullptr, r,
                                   s, 3)))
            return st;
    }
    // dX = dY W' + (sV) A
    TcParams prm{};
    prm.M = M;
    prm.Nd = K;
    prm.w_cols = K;
    prm.nk_main = cdiv(N, kGemmBK);
    prm.lora_steps = rp / 64;
    prm.r = r;
    prm.tab = w.tab;
    prm.ncg = prm.nkg = 1;
    prm.cg_first[1] = cdiv(K, PairCfg::BN);
    prm.kg_first[1] = prm.nk_main;
    prm.pj[0] = TcProj{w.q, w.s2, w.mean, w.absmax, N, static_cast<uint16_t *>(dX), K, K, 0, 0};
    prm.flags = b.sk.flags;
    prm.slots = b.sk.slots;
    prm.wait_ns = wait_ns();
    prm.kernel_id = 2;
    GemmMaps gm;
    memset(&gm, 0, sizeof gm);
    gm.act[0] = tmD;
    gm.codes[0] = tmC;
    gm.lact = tmV;
    gm.lw[0] = tmA;
    if ((st = launch_gemm<kDx>(gm, prm, s))) return st;
    // dA = (sV)^T X (rows k of dA^T) and dB = s dY^T U (rows n), both
    // contracting over the M tokens, in one launch
    const SkJob ja{&tmXmn, &tmVmn, sk_plan(K, M, r), kRedDA, 1.0f, nullptr, 0, nullptr, 0, dA};
    const SkJob jb{&tmDmn, &tmUp, sk_plan(N, M, r), kRedDB, scale, nullptr, 0, nullptr, 0, dB};
    if ((st = run_skinny<1, 1>(ja, &jb, r, s, 5))) return st;
    return ok();
}

qlora_status qlora_linear_fwd(const void *X, int64_t M, const qlora_nf4_weight *w, const void *A, const void *B,
                              int r, float scale, void *Y, void *U_save, void *ws, size_t ws_bytes,
                              qlora_stream_t stream) {
    if (!w) return fail(QLORA_ERR_NULL, "weight descriptor is NULL");
    return linear_fwd_impl(X, M, wt_of(w), A, B, r, scale, Y, U_save, ws, ws_bytes, stream, r);
}

qlora_status qlora_q4_linear_fwd(const void *X, int64_t M, const qlora_q4_weight *w, const void *A, const void *B,
                                 int r, float scale, void *Y, void *U_save, void *ws, size_t ws_bytes,
                                 qlora_stream_t stream) {
    if (!w) return fail(QLORA_ERR_NULL, "weight descriptor is NULL");
    return linear_fwd_impl(X, M, wt_of(w), A, B, r, scale, Y, U_save, ws, ws_bytes, stream, r);
}

qlora_status qlora_linear_bwd(const void *dY, const void *X, const void *U_saved, int64_t M,
                              const qlora_nf4_weight *w, const void *A, const void *B, int r, float scale, void *dX,
                              float *dA, float *dB, void *ws, size_t ws_bytes, qlora_stream_t stream) {
    if (!w) return fail(QLORA_ERR_NULL, "weight descriptor is NULL");
    return linear_bwd_impl(dY, X, U_saved, M, wt_of(w), A, B, r, scale, dX, dA, dB, ws, ws_bytes, stream, r);
}

qlora_status qlora_q4_linear_bwd(const void *dY, const void *X, const void *U_saved, int64_t M,
                                 const qlora_q4_weight *w, const void *A, const void *B, int r, float scale, void *dX,
                                 float *dA, float *dB, void *ws, size_t ws_bytes, qlora_stream_t stream) {
    if (!w) return fail(QLORA_ERR_NULL, "weight descriptor is NULL");
    return linear_bwd_impl(dY, X, U_saved, M, wt_of(w), A, B, r, scale, dX, dA, dB, ws, ws_bytes, stream, r);
}

// ---- projection groups ------------------------------------------------------

static_assert(QLORA_MAX_GROUP == kMaxGroup, "group size of the ABI and of the kernels");

// Validated view of a group's projections.
struct GroupView {
    int n;
    int64_t K;
    Wt w[kMaxGroup];
};

// outputs: also check the pointers the call reads or writes besides the
// weights and adapters (not for the workspace queries).
static qlora_status check_group(int64_t M, const qlora_proj *proj, int n, int r, bool bwd, GroupView &gv,
                                bool outputs = true) {
    if (!proj) return fail(QLORA_ERR_NULL, "projection list is NULL");
    if (n < 1 || n > kMaxGroup) return fail(QLORA_ERR_SHAPE, "group of %d projections: need 1..%d", n, kMaxGroup);
    if (r < 8 || r > 128 || r % 8) return fail(QLORA_ERR_RANK, "group rank r = %d: need 8 <= r <= 128, r %% 8 == 0", r);
    if (M < 0 || M >= kMaxDim) return fail(QLORA_ERR_SHAPE, "M = %lld out of range", (long long)M);
    gv.n = n;
    for (int g = 0; g < n; ++g) {
        const qlora_proj &pj = proj[g];
        if (!pj.w) return fail(QLORA_ERR_NULL, "projection %d: weight descriptor is NULL", g);
        gv.w[g] = wt_of(pj.w);
        qlora_status st = check_weight(gv.w[g], true);
        if (st) return st;
        if (g == 0) gv.K = gv.w[0].cols;
        if (gv.w[g].cols != gv.K)
            return fail(QLORA_ERR_SHAPE, "projection %d has K = %lld, projection 0 K = %lld", g,
                        (long long)gv.w[g].cols, (long long)gv.K);
        if (!pj.A || !pj.B) return fail(QLORA_ERR_NULL, "projection %d: A or B is NULL", g);
        if (!al16(pj.A) || !al16(pj.B)) return fail(QLORA_ERR_ALIGN, "projection %d: A and B must be 16-byte aligned", g);
        if (M == 0 || !outputs) continue;
        if (!bwd) {
            if (!pj.Y) return fail(QLORA_ERR_NULL, "projection %d: Y is NULL", g);
            if (!al16(pj.Y)) return fail(QLORA_ERR_ALIGN, "projection %d: Y must be 16-byte aligned", g);
        } else {
            if (!pj.dY) return fail(QLORA_ERR_NULL, "projection %d: dY is NULL", g);
            if (!al16(pj.dY)) return fail(QLORA_ERR_ALIGN, "projection %d: dY must be 16-byte aligned", g);
        }
    }
    if (bwd && outputs)
        for (int g = 0; g < n; ++g) {
            if (!proj[g].dA || !proj[g].dB) return fail(QLORA_ERR_NULL, "projection %d: dA or dB is NULL", g);
            if (!al16(proj[g].dA) || !al16(proj[g].dB))
                return fail(QLORA_ERR_ALIGN, "projection %d: dA and dB must be 16-byte aligned", g);
        }
    return QLORA_OK;
}

// The tensor-core paths of a group: forward beyond the few-token sizes,
// backward from kTcMinM tokens with every N_g a multiple of 8. Otherwise the
// projections run one by one through the single-layer paths.
static bool group_tc_fwd(int64_t M) { return M > kSmallMaxM; }
static bool group_tc_bwd(int64_t M, const GroupView &gv) {
    if (M < kTcMinM) return false;
    for (int g = 0; g < gv.n; ++g)
        if (gv.w[g].rows % 8) return false;
    return true;
}

struct GroupWs {
    uint16_t *Acat, *sU, *sV, *U, *parts;
    float *dAcat;
    float *few_slots;
    uint32_t *few_counters;
    SkArea sk;
    char *rest;  // per-projection workspace of the one-by-one paths
    size_t rest_bytes;
};
// A group's few-token forward runs as one launch over all its projections
// when each of them takes the few-token kernel.
static bool group_few_fwd(int64_t M, const GroupView &gv) {
    for (int g = 0; g < gv.n; ++g)
        if (!few_path(M, gv.w[g].rows, gv.K)) return false;
    return true;
}
static int64_t group_tiles(const GroupView &gv) {
    int64_t t = 0;
    for (int g = 0; g < gv.n; ++g) t += cdiv(gv.w[g].rows, FewCfg::ROWS);
    return t;
}
static size_t group_ws(int64_t M, const GroupView &gv, int r, bool bwd, void *ws, size_t ws_bytes, GroupWs *out) {
    const int n = gv.n;
    const int64_t K = gv.K, R = (int64_t)n * r;
    Carve c(ws);
    GroupWs w{};
    size_t per = 0;
    if (!bwd && group_tc_fwd(M)) {
        w.Acat = c.take<uint16_t>((size_t)(R * K));
        w.sU = c.take<uint16_t>((size_t)(M * R));
        w.sk = take_sk_area(c);
    } else if (!bwd && group_few_fwd(M, gv)) {
        const FewPlan fp = few_plan_tiles(M, group_tiles(gv), K);
        w.sU = c.take<uint16_t>((size_t)M * n * lora_pad(r));
        w.few_slots = c.take<float>((size_t)fp.warps * few_slot_floats(M));
        w.few_counters = c.take<uint32_t>((size_t)fp.tiles);
    } else if (bwd && group_tc_bwd(M, gv)) {
        w.Acat = c.take<uint16_t>((size_t)(R * K));
        w.sV = c.take<uint16_t>((size_t)(M * R));
        w.U = c.take<uint16_t>((size_t)(M * R));
        w.dAcat = c.take<float>((size_t)(R * K));
        w.sk = take_sk_area(c);
    } else {
        if (bwd) w.parts = c.take<uint16_t>((size_t)(n * M * K));
        for (int g = 0; g < n; ++g)
            per = std::max(per, bwd ? bwd_ws(M, gv.w[g].rows, K, r, nullptr, nullptr)
                                    : fwd_ws(M, gv.w[g].rows, K, r, nullptr, nullptr));
        w.rest = c.take<char>(per);
    }
    const size_t need = c.off;
    w.rest_bytes = per;
    if (out) *out = w;
    (void)ws_bytes;
    return need;
}

// The stacked A_g [n * r, K]: the caller's when they already lie back to
// back, else a copy in the workspace.
static qlora_status stack_A(const qlora_proj *proj, int n, int r, int64_t K, uint16_t *Acat, cudaStream_t s,
                            const void **out) {
    const size_t bytes = (size_t)r * (size_t)K * 2;
    bool contiguous = true;
    for (int g = 1; g < n; ++g)
        contiguous = contiguous && static_cast<const char *>(proj[g].A) == static_cast<const char *>(proj[0].A) + g * bytes;
    if (contiguous) {
        *out = proj[0].A;
        return QLORA_OK;
    }
    for (int g = 0; g < n; ++g)
        if (cudaMemcpyAsync(reinterpret_cast<char *>(Acat) + g * bytes, proj[g].A, bytes, cudaMemcpyDeviceToDevice,
                            s) != cudaSuccess)
            return fail(QLORA_ERR_CUDA, "copying A of projection %d failed", g);
    *out = Acat;
    return QLORA_OK;
}

static qlora_status group_fwd_impl(const void *X, int64_t M, const qlora_proj *proj, int n, int r, float scale,
                                   void *U_save, void *ws, size_t ws_bytes, qlora_stream_t stream) {
    GroupView gv;
    qlora_status st = check_group(M, proj, n, r, false, gv);
    if (st) return st;
    if (M > 0 && !X) return fail(QLORA_ERR_NULL, "X is NULL");
    if ((X && !al16(X)) || (U_save && !al16(U_save)) || (ws && !al16(ws)))
        return fail(QLORA_ERR_ALIGN, "X, U_save and the workspace must be 16-byte aligned");
    if (M == 0) return ok();
    GroupWs gw;
    const size_t need = group_ws(M, gv, r, false, ws, ws_bytes, &gw);
    if (!ws) return fail(QLORA_ERR_NULL, "workspace is NULL");
    if (ws_bytes < need) return fail(QLORA_ERR_WORKSPACE, "group forward workspace %zu < %zu bytes", ws_bytes, need);
    const int64_t K = gv.K, R = (int64_t)n * r;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (group_few_fwd(M, gv)) {
        // few tokens: one HBM-bound launch over the row tiles of every projection
        const Wt *wp[kMaxGroup];
        const void *Ap[kMaxGroup], *Bp[kMaxGroup];
        void *Yp[kMaxGroup];
        for (int g = 0; g < n; ++g) {
            wp[g] = &gv.w[g];
            Ap[g] = proj[g].A;
            Bp[g] = proj[g].B;
            Yp[g] = proj[g].Y;
        }
        return few_fwd_launch(static_cast<const uint16_t *>(X), M, wp, Ap, Bp, Yp, n, r, scale,
                              static_cast<uint16_t *>(U_save), (int)R, gw.sU, lora_pad(r), gw.few_slots,
                              gw.few_counters, s);
    }
    if (!group_tc_fwd(M)) {
        // few tokens: the projections one by one (HBM-bound kernels)
        for (int g = 0; g < n; ++g)
            if ((st = linear_fwd_impl(X, M, gv.w[g], proj[g].A, proj[g].B, r, scale, proj[g].Y,
                                      U_save ? static_cast<uint16_t *>(U_save) + g * r : nullptr, gw.rest,
                                      gw.rest_bytes, stream, (int)R)))
                return st;
        return ok();
    }
    if ((st = tc_device_ok()) || (st = tc_setup<kFwd>())) return st;
    const void *Acat;
    if ((st = stack_A(proj, n, r, K, gw.Acat, s, &Acat))) return st;
    GemmMaps gm;
    memset(&gm, 0, sizeof gm);
    CUtensorMap tmAc;
    if ((st = make_map(&gm.act[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, K, M, K * 2, 64, 128,
                       CU_TENSOR_MAP_SWIZZLE_128B, "X")) ||
        (st = make_map(&tmAc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Acat, K, R, K * 2, 64, 64,
                       CU_TENSOR_MAP_SWIZZLE_128B, "stacked A")) ||
        (st = make_map(&gm.lact, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, gw.sU, R, M, R * 2, 64, 128,
                       CU_TENSOR_MAP_SWIZZLE_128B, "sU")))
        return st;
    TcParams prm{};
    prm.M = M;
    prm.w_cols = K;
    prm.nk_main = K / kGemmBK;
    prm.lora_steps = (int)cdiv(r, 64);
    prm.r = r;
    prm.tab = kTableNF4;
    prm.ncg = n;
    prm.nkg = 1;
    prm.kg_first[1] = prm.nk_main;
    for (int g = 0; g < n; ++g) {
        const int64_t N = gv.w[g].rows;
        if ((st = make_map(&gm.codes[g], CU_TENSOR_MAP_DATA_TYPE_UINT8, gv.w[g].codes, K / 2, N, K / 2, 32, 128,
                           CU_TENSOR_MAP_SWIZZLE_32B, "codes")) ||
            (st = make_map(&gm.lw[g], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, proj[g].B, r, N, r * 2, 64, 128,
                           CU_TENSOR_MAP_SWIZZLE_128B, "B")))
            return st;
        prm.cg_first[g + 1] = prm.cg_first[g] + cdiv(N, PairCfg::BN);
        prm.pj[g] = TcProj{gv.w[g].q, gv.w[g].s2, gv.w[g].mean, gv.w[g].absmax, N, static_cast<uint16_t *>(proj[g].Y),
                           N, N, g * r, 0};
    }
    prm.Nd = prm.cg_first[n] * PairCfg::BN;
    // U_g = X A_g^T for all projections in one pass: U to U_save, s*U to the workspace
    if ((st = run_skinny<0, 0>(SkJob{&gm.act[0], &tmAc, sk_plan(M, K, (int)R), kRedU, scale,
                                     static_cast<uint16_t *>(U_save), (int)R, gw.sU, (int)R, nullptr},
                               nullptr, (int)R, s, 3, gw.sk.flags, kSkFlagWords)))
        return st;
    prm.flags = gw.sk.flags;
    prm.slots = gw.sk.slots;
    prm.wait_ns = wait_ns();
    prm.kernel_id = 1;
    if ((st = launch_gemm<kFwd>(gm, prm, s))) return st;
    return ok();
}

static qlora_status group_bwd_impl(const void *X, const void *U_saved, int64_t M, const qlora_proj *proj, int n, int r,
                                   float scale, void *dX, void *ws, size_t ws_bytes, qlora_stream_t stream) {
    GroupView gv;
    qlora_status st = check_group(M, proj, n, r, true, gv);
    if (st) return st;
    if (M > 0 && (!X || !dX)) return fail(QLORA_ERR_NULL, "X or dX is NULL");
    if ((X && !al16(X)) || (dX && !al16(dX)) || (U_saved && !al16(U_saved)) || (ws && !al16(ws)))
        return fail(QLORA_ERR_ALIGN, "X, U_saved, dX and the workspace must be 16-byte aligned");
    const int64_t K = gv.K, R = (int64_t)n * r;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (M == 0) {
        for (int g = 0; g < n; ++g)
            if (cudaMemsetAsync(proj[g].dA, 0, sizeof(float) * r * K, s) != cudaSuccess ||
                cudaMemsetAsync(proj[g].dB, 0, sizeof(float) * r * gv.w[g].rows, s) != cudaSuccess)
                return fail(QLORA_ERR_CUDA, "memset of dA/dB failed");
        return ok();
    }
    GroupWs gw;
    const size_t need = group_ws(M, gv, r, true, ws, ws_bytes, &gw);
    if (!ws) return fail(QLORA_ERR_NULL, "workspace is NULL");
    if (ws_bytes < need) return fail(QLORA_ERR_WORKSPACE, "group backward workspace %zu < %zu bytes", ws_bytes, need);
    const uint16_t *U16 = static_cast<const uint16_t *>(U_saved);
    if (!group_tc_bwd(M, gv)) {
        // few tokens: the projections one by one, then dX = the sum of their parts
        for (int g = 0; g < n; ++g)
            if ((st = linear_bwd_impl(proj[g].dY, X, U16 ? U16 + g * r : nullptr, M, gv.w[g], proj[g].A, proj[g].B, r,
                                      scale, gw.parts + g * M * K, proj[g].dA, proj[g].dB, gw.rest, gw.rest_bytes,
                                      stream, (int)R)))
                return st;
        {
            ProfScope ps(QLORA_KERNEL_DX_SIMT, s);
            k_sum_parts<<<(unsigned)cdiv(M * K / 8, 256), 256, 0, s>>>(gw.parts, n, M * K,
                                                                      static_cast<uint16_t *>(dX));
        }
        if ((st = launch_check("k_sum_parts"))) return st;
        return ok();
    }
    if ((st = tc_device_ok()) || (st = tc_setup<kDx>())) return st;
    const void *Acat;
    if ((st = stack_A(proj, n, r, K, gw.Acat, s, &Acat))) return st;
    const uint16_t *Ucur = U16 ? U16 : gw.U;
    GemmMaps gm;
    memset(&gm, 0, sizeof gm);
    CUtensorMap tmDmn[kMaxGroup], tmBp[kMaxGroup], tmUg[kMaxGroup], tmXk, tmXmn, tmVmn;
    if ((st = make_map(&tmXk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, K, M, K * 2, 64, 128,
                       CU_TENSOR_MAP_SWIZZLE_128B, "X")) ||
        (st = make_map(&tmXmn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, K, M, K * 2, 64, 64,
                       CU_TENSOR_MAP_SWIZZLE_128B, "X (MN)")) ||
        (st = make_map(&gm.lact, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, gw.sV, R, M, R * 2, 64, 128,
                       CU_TENSOR_MAP_SWIZZLE_128B, "sV")) ||
        (st = make_map(&tmVmn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, gw.sV, R, M, R * 2, 64, 64,
                       CU_TENSOR_MAP_SWIZZLE_128B, "sV (MN)")) ||
        (st = make_map(&gm.lw[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Acat, K, R, K * 2, 64, 64,
                       CU_TENSOR_MAP_SWIZZLE_128B, "stacked A")))
        return st;
    TcParams prm{};
    prm.M = M;
    prm.Nd = K;
    prm.w_cols = K;
    prm.tab = kTableNF4;
    prm.ncg = 1;
    prm.nkg = n;
    prm.cg_first[1] = cdiv(K, PairCfg::BN);
    SkJob vj[kMaxGroup], bj[kMaxGroup];
    for (int g = 0; g < n; ++g) {
        const int64_t N = gv.w[g].rows;
        if ((st = make_map(&gm.act[g], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, proj[g].dY, N, M, N * 2, 64, 128,
                           CU_TENSOR_MAP_SWIZZLE_128B, "dY")) ||
            (st = make_map(&tmDmn[g], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, proj[g].dY, N, M, N * 2, 64, 64,
                           CU_TENSOR_MAP_SWIZZLE_128B, "dY (MN)")) ||
            (st = make_map(&gm.codes[g], CU_TENSOR_MAP_DATA_TYPE_UINT8, gv.w[g].codes, K / 2, N, K / 2, 64, 64,
                           CU_TENSOR_MAP_SWIZZLE_64B, "codes")) ||
            (st = make_map(&tmBp[g], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, proj[g].B, r, N, r * 2, 64, 64,
                           CU_TENSOR_MAP_SWIZZLE_128B, "B")) ||
            (st = make_map(&tmUg[g], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Ucur + g * r, r, M, R * 2, 64, 64,
                           CU_TENSOR_MAP_SWIZZLE_128B, "U")))
            return st;
        prm.kg_first[g + 1] = prm.kg_first[g] + cdiv(N, kGemmBK);
        prm.pj[g] = TcProj{gv.w[g].q, gv.w[g].s2, gv.w[g].mean, gv.w[g].absmax, N, static_cast<uint16_t *>(dX), K,
                           K, 0, 0};
        // V_g = dY_g B_g -> columns [g r, (g + 1) r) of sV = bf16(s * V)
        vj[g] = SkJob{&gm.act[g], &tmBp[g], sk_plan(M, N, r), kRedV, scale, nullptr, 0, gw.sV + g * r, (int)R, nullptr};
        vj[g].zend = r;
        // dB_g = s dY_g^T U_g
        bj[g] = SkJob{&tmDmn[g], &tmUg[g], sk_plan(N, M, r), kRedDB, scale, nullptr, 0, nullptr, 0, proj[g].dB};
    }
    prm.nk_main = prm.kg_first[n];
    prm.lora_steps = (int)cdiv(R, 64);
    prm.r = (int)R;
    int rsv[kSkMaxJobs];
    for (int g = 0; g < kSkMaxJobs; ++g) rsv[g] = r;
    // every projection's V in one launch
    if ((st = run_skinny_jobs<0, 1>(vj, rsv, n, s, 4, gw.sk.flags, kSkFlagWords))) return st;
    if (!U16) {
        // U recomputed for all projections in one pass as X A^T (A stacked)
        if ((st = run_skinny<0, 0>(SkJob{&tmXk, &gm.lw[0], sk_plan(M, K, (int)R), kRedV, 1.0f, nullptr, 0, gw.U,
                                         (int)R, nullptr},
                                   nullptr, (int)R, s, 3)))
            return st;
    }
    // dX = sum_g dY_g W_g' + (sV) A over all projections' rows in one launch
    prm.flags = gw.sk.flags;
    prm.slots = gw.sk.slots;
    prm.wait_ns = wait_ns();
    prm.kernel_id = 2;
    if ((st = launch_gemm<kDx>(gm, prm, s))) return st;
    // dA of all projections at once: dA^T = X^T (sV), rank n r; into the
    // caller's dA when those lie back to back
    const size_t abytes = (size_t)r * (size_t)K * sizeof(float);
    bool dA_contiguous = true;
    for (int g = 1; g < n; ++g)
        dA_contiguous = dA_contiguous &&
                        reinterpret_cast<char *>(proj[g].dA) == reinterpret_cast<char *>(proj[0].dA) + g * abytes;
    float *dAdst = dA_contiguous ? proj[0].dA : gw.dAcat;
    // dA of all projections (rank n r) and every projection's dB in one
    // launch when their ranks take the same number of 64-wide tiles, else dA
    // in one launch and the dB in another
    SkJob gj[kSkMaxJobs];
    int rsg[kSkMaxJobs];
    gj[0] = SkJob{&tmXmn, &tmVmn, sk_plan(K, M, (int)R), kRedDA, 1.0f, nullptr, 0, nullptr, 0, dAdst};
    rsg[0] = (int)R;
    const bool together = gj[0].pl.zt == bj[0].pl.zt && n + 1 <= kSkMaxJobs;
    if (together) {
        for (int g = 0; g < n; ++g) {
            gj[1 + g] = bj[g];
            rsg[1 + g] = r;
        }
        if ((st = run_skinny_jobs<1, 1>(gj, rsg, n + 1, s, 5))) return st;
    } else {
        if ((st = run_skinny_jobs<1, 1>(gj, rsg, 1, s, 5))) return st;
        if ((st = run_skinny_jobs<1, 1>(bj, rsv, n, s, 5))) return st;
    }
    if (!dA_contiguous)
        for (int g = 0; g < n; ++g)
            if (cudaMemcpyAsync(proj[g].dA, reinterpret_cast<char *>(gw.dAcat) + g * abytes, abytes,
                                cudaMemcpyDeviceToDevice, s) != cudaSuccess)
                return fail(QLORA_ERR_CUDA, "copying dA of projection %d failed", g);
    return ok();
}

size_t qlora_group_fwd_workspace(int64_t M, const qlora_proj *proj, int n, int r) {
    GroupView gv;
    if (check_group(M, proj, n, r, false, gv, false) != QLORA_OK) return 0;
    return group_ws(M, gv, r, false, nullptr, 0, nullptr);
}

size_t qlora_group_bwd_workspace(int64_t M, const qlora_proj *proj, int n, int r) {
    GroupView gv;
    if (check_group(M, proj, n, r, true, gv, false) != QLORA_OK) return 0;
    return group_ws(M, gv, r, true, nullptr, 0, nullptr);
}

qlora_status qlora_group_fwd(const void *X, int64_t M, const qlora_proj *proj, int n, int r, float scale,
                             void *U_save, void *ws, size_t ws_bytes, qlora_stream_t stream) {
    return group_fwd_impl(X, M, proj, n, r, scale, U_save, ws, ws_bytes, stream);
}

qlora_status qlora_group_bwd(const void *X, const void *U_saved, int64_t M, const qlora_proj *proj, int n, int r,
                             float scale, void *dX, void *ws, size_t ws_bytes, qlora_stream_t stream) {
    return group_bwd_impl(X, U_saved, M, proj, n, r, scale, dX, ws, ws_bytes, stream);
}

void qlora_q4_table(int table, float levels[16]) {
    if (!levels) return;
    static const float tabs[2][16] = {QLORA_NF4_LEVELS, QLORA_INT4_LEVELS};
    const bool known = table == QLORA_TABLE_NF4 || table == QLORA_TABLE_INT4;
    for (int i = 0; i < 16; ++i) levels[i] = known ? tabs[table][i] : 0.0f;
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
