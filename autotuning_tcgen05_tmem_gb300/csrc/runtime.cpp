// Plans, launches, the on-device tuner and the tune-once cache.
//
// Sources (page title, section):
//  * "Tile Selection: Cost Models Against Measurement", "Measurement, and what it
//    must control": interleave candidates (clock drift), realistic input values,
//    many repetitions per timing (launch overhead); results cached by shape,
//    dtype, device model and library version.  "Hybrid strategies": resource
//    filter -> model rank -> measure the top handful.
//  * "Autotuning & cost models" §4: benchmark on the first call for a key,
//    remember the winner, reuse it for every later call with the same key.
//  * "CuTile Autotuning": tune once, cache config and launchable object, launch
//    directly; the search space includes the original fixed config; in-place
//    kernels are tuned on separate buffers (here: tuning never touches user
//    memory); DISABLE_AUTOTUNE-style switch for correctness runs.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <map>
#include <mutex>
#include <numeric>
#include <string>
#include <vector>

#include "gemm_internal.h"
#include "schedule.h"

namespace gemmgb {

std::atomic<int64_t> g_timeout_ns{2000000000LL};
std::atomic<int32_t> g_debug_stall{0};
// How B reaches the tensor cores: 0 = by dtype (bf16 read MN-major in place;
// FP8 too when N % 16 == 0; fp32 transposed to a K-major copy), 1 = always
// transposed, 2 = always MN-major.
std::atomic<int32_t> g_b_route{0};
// How split-K slices exchange partial tiles: 0 = through distributed shared
// memory when all units fit in one wave and the slices of a tile can form a
// cluster, else global memory; 1 = always global memory.
std::atomic<int32_t> g_split_route{0};
// How long (SM clock cycles) the owner of a one-wave split-K share waits for
// the other slices before it hands the share over: about 25 us at the top
// clock.  0 makes every owner hand over at once (tests drive that path).
std::atomic<int64_t> g_share_poll{50000};
// Value distribution of the tuner's synthetic operands: 1 = normal with
// standard deviation 1/sqrt(K) (the default: the workloads' N(0,1)/sqrt(K)
// family), 0 = uniform of the same standard deviation.
std::atomic<int32_t> g_tune_fill{1};
// Operands read with one tensor copy per stage where the layout allows (1), or
// one copy per 128-byte span (0), in plans made from now on.
std::atomic<int32_t> g_span3d{1};
// Checked runs (GEMM_CHECK set to anything but 0 in the environment, or
// gemm_debug_set(4, 1)): every run synchronises its stream and reports a
// device-side timeout itself instead of leaving it to gemm_plan_status.
static int32_t check_from_env()
{
    const char *v = getenv("GEMM_CHECK");
    return (v && *v && strcmp(v, "0") != 0) ? 1 : 0;
}
std::atomic<int32_t> g_check{check_from_env()};

// ---------------------------------------------------------------------------
// TMA descriptor encoding through the driver entry point
// ---------------------------------------------------------------------------

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;

static int encoder_ready()
{
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

// Row-major [outer, inner] matrix, box [box_outer, box_inner].
static int encode_2d(CUtensorMap *m, int dt, const void *ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
                     uint32_t box_outer, CUtensorMapSwizzle sw, CUtensorMapL2promotion l2)
{
    if (!encoder_ready()) return set_error(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * (uint64_t)elt_bytes(dt)};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType t = dt == GEMM_BF16       ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                  : is_fp8(dt)          ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    CUresult r = g_encode(m, t, 2, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          sw, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return set_error(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for [%llu x %llu] box [%u x %u]", (int)r,
                         (unsigned long long)outer, (unsigned long long)inner, box_outer, box_inner);
    return GEMM_OK;
}

// The same [outer][inner] matrix seen in 3-D as [inner / span][outer][span]
// (inner a whole number of spans): a box of [n_spans][box_outer][span] takes a
// stage's consecutive spans in one copy and lands them span after span, as
// n_spans two-dimensional copies of [box_outer][span] would.
static int encode_spans(CUtensorMap *m, int dt, const void *ptr, uint64_t inner, uint64_t outer, uint32_t span,
                        uint32_t box_outer, uint32_t n_spans)
{
    if (!encoder_ready()) return set_error(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const uint64_t e = (uint64_t)elt_bytes(dt);
    const cuuint64_t dims[3] = {span, outer, inner / span};
    const cuuint64_t strides[2] = {inner * e, span * e};
    const cuuint32_t box[3] = {span, box_outer, n_spans};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType t = dt == GEMM_BF16       ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                  : is_fp8(dt)          ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                        : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    CUresult r = g_encode(m, t, 3, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return set_error(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for [%llu x %llu] in spans, box [%u x %u x %u]",
                         (int)r, (unsigned long long)outer, (unsigned long long)inner, n_spans, box_outer, span);
    return GEMM_OK;
}

static int cuda_err(cudaError_t e, const char *what)
{
    return set_error(GEMM_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// ---------------------------------------------------------------------------
// Device parameters
// ---------------------------------------------------------------------------

static double env_double(const char *name, double dflt)
{
    const char *v = getenv(name);
    if (!v || !*v) return dflt;
    char *end = nullptr;
    const double x = strtod(v, &end);
    return (end && end != v && x > 0) ? x : dflt;
}

int model_params_load(const char *path, gemm_device_params *out)
{
    if (!path || !out) return set_error(GEMM_ERR_INVALID_ARG, "null path or parameters");
    FILE *f = fopen(path, "r");
    if (!f) return set_error(GEMM_ERR_INVALID_ARG, "cannot read model parameters from %s", path);
    gemm_device_params d = *out;
    struct Field { const char *name; double *dst; };
    const Field fields[] = {{"peak_tflops_bf16", &d.peak_tflops_bf16}, {"peak_tflops_tf32", &d.peak_tflops_tf32},
                            {"peak_tflops_fp8", &d.peak_tflops_fp8},   {"hbm_gbs", &d.hbm_gbs},
                            {"sm_clock_mhz", &d.sm_clock_mhz},         {"l2_gbs", &d.l2_gbs},
                            {"mma_issue_clk", &d.mma_issue_clk},       {"kblock_clk", &d.kblock_clk},
                            {"mem_latency_us", &d.mem_latency_us},     {"epi_elems_per_clk", &d.epi_elems_per_clk},
                            {"epi_gelu_elems_per_clk", &d.epi_gelu_elems_per_clk},
                            {"splitk_gbs", &d.splitk_gbs},             {"launch_us", &d.launch_us}};
    char line[512];
    int lineno = 0, rc = GEMM_OK;
    while (rc == GEMM_OK && fgets(line, sizeof line, f)) {
        ++lineno;
        char *hash = strchr(line, '#');
        if (hash) *hash = 0;
        char name[128];
        double value = 0.0;
        char extra[8];
        const int got = sscanf(line, "%127s %lf %7s", name, &value, extra);
        if (got <= 0) continue;                      // blank or comment
        if (got != 2 || !(value > 0.0) || !isfinite(value)) {
            rc = set_error(GEMM_ERR_INVALID_ARG, "%s:%d: expected \"name positive-value\"", path, lineno);
            break;
        }
        bool known = false;
        for (const Field &fd : fields)
            if (strcmp(fd.name, name) == 0) {
                *fd.dst = value;
                known = true;
            }
        if (!known) rc = set_error(GEMM_ERR_INVALID_ARG, "%s:%d: unknown model parameter %s", path, lineno, name);
    }
    fclose(f);
    if (rc == GEMM_OK) *out = d;
    return rc;
}

int query_params(gemm_device_params *d)
{
    params_default(d);
    int dev = 0, v = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return set_error(GEMM_ERR_NO_DEVICE, "no CUDA device: %s", cudaGetErrorString(e));
    }
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return cuda_err(e, "cudaDeviceGetAttribute(SM count)");
    d->sm_count = v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess) d->smem_per_block = v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) == cudaSuccess) d->l2_bytes = v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrClockRate, dev) == cudaSuccess && v > 0) d->sm_clock_mhz = v / 1000.0;
    int regs = 0;
    if (kernel_attributes(GEMM_BF16, &regs, nullptr) == cudaSuccess) d->kernel_regs = regs;
    d->peak_tflops_bf16 = env_double("GEMM_PEAK_BF16_TFLOPS", d->peak_tflops_bf16);
    d->peak_tflops_tf32 = env_double("GEMM_PEAK_TF32_TFLOPS", d->peak_tflops_bf16 / 2.0);
    d->peak_tflops_fp8 = env_double("GEMM_PEAK_FP8_TFLOPS", d->peak_tflops_bf16 * 2.0);
    d->hbm_gbs = env_double("GEMM_HBM_GBS", d->hbm_gbs);
    const char *mp = getenv("GEMM_MODEL_PARAMS");
    if (mp && *mp) return model_params_load(mp, d);
    return GEMM_OK;
}

static int check_device_arch(int *device_out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return set_error(GEMM_ERR_NO_DEVICE, "no CUDA device: %s", cudaGetErrorString(e));
    }
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3)
        return set_error(GEMM_ERR_UNSUPPORTED, "kernels are built for sm_103a; device %d is sm_%d%d", dev, major, minor);
    if (device_out) *device_out = dev;
    return GEMM_OK;
}

}  // namespace gemmgb

// ---------------------------------------------------------------------------
// Plan object
// ---------------------------------------------------------------------------

struct DescEntry {
    const void *a = nullptr, *b = nullptr, *sa = nullptr, *sb = nullptr;
    void *c = nullptr;
    bool valid = false;
    CUtensorMap ma, mb, mc, msa, msb;   // msa, msb: MX scales (block-scaled plans only)
};

struct gemm_plan_s {
    int64_t M = 0, N = 0, K = 0;
    int dt = 0, epi = 0, device = 0;
    gemm_config cfg{};
    gemm_device_params dev{};
    gemmgb::Layout L{};
    gemmgb::KernelParams kp{};
    int grid = 0, smem_request = 0;
    float *workspace = nullptr;
    bool owns_workspace = false;
    int32_t *aux = nullptr;          // [0] status word, [1..n_counters] split-K counters
    uint64_t *epochs = nullptr;      // one-wave split-K: arrival counts per tile share (only ever grow)
    int64_t n_counters = 0;
    int64_t tiles = 0;
    std::vector<DescEntry> descs = std::vector<DescEntry>(16);
    int next_desc = 0;
    void *hA = nullptr, *hB = nullptr, *hBias = nullptr, *hC = nullptr;  // device buffers for run_host
    bool b_kmajor = false;           // B is first transposed into bt ([N, K], K contiguous)
    int32_t independent = 0;         // GEMM_OPERAND_A | GEMM_OPERAND_B: operands that the work
                                     // queued before a launch never writes
    void *bt = nullptr;
    // Host-buffer batches (run_host_many): a second plan of the same
    // configuration (its own split-K workspace, counters and device buffers)
    // and a second stream, so that one GEMM's copies overlap the other's kernel.
    gemm_plan_s *twin = nullptr;
    cudaStream_t side = nullptr;
};

namespace gemmgb {

static int configure_smem_limit(int dt, int64_t bytes)
{
    static std::mutex mu;
    static std::map<std::pair<int, int>, int64_t> done;  // (device, dtype) -> bytes set
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lk(mu);
    auto key = std::make_pair(dev, dt);
    auto it = done.find(key);
    if (it != done.end() && it->second >= bytes) return GEMM_OK;
    cudaError_t e = set_kernel_smem_limit(dt, (int)bytes);
    if (e != cudaSuccess) return cuda_err(e, "cudaFuncSetAttribute(max dynamic shared memory)");
    done[key] = bytes;
    return GEMM_OK;
}

static bool valid_enums(int dt, int epi)
{
    return dt >= GEMM_BF16 && dt <= GEMM_MXFP8_E4M3 && epi >= GEMM_EPI_NONE && epi <= GEMM_EPI_BIAS_SWIGLU;
}

// Residual epilogues are the bias / ReLU / GELU ones followed by "+ R".
static bool has_residual(int epi) { return is_residual(epi); }
// The kernel's epilogue code: 0 none, 1 bias, 2 ReLU, 3 GELU, and the gated
// 7 ReGLU, 8 GeGLU, 9 SwiGLU; the residual is a run argument.
static int act_code(int epi) { return has_residual(epi) ? epi - 3 : epi; }

static int check_extents(int64_t M, int64_t N, int64_t K)
{
    const int64_t lim = (int64_t)1 << 31;
    if (M < 0 || N < 0 || K < 0 || M >= lim || N >= lim || K >= lim)
        return set_error(GEMM_ERR_INVALID_ARG, "extents must be in [0, 2^31): M=%lld N=%lld K=%lld", (long long)M,
                         (long long)N, (long long)K);
    return GEMM_OK;
}

void destroy_plan(gemm_plan_t p);

// Builds a plan; `shared_ws` (may be null) is a caller-owned split-K workspace
// of at least the needed size (used while tuning many candidates).
int make_plan(int64_t M, int64_t N, int64_t K, int dt, int epi, const gemm_config &cfg,
              const gemm_device_params &dev, float *shared_ws, gemm_plan_t *out)
{
    *out = nullptr;
    int rc = check_extents(M, N, K);
    if (rc) return rc;
    if (!valid_enums(dt, epi)) return set_error(GEMM_ERR_INVALID_ARG, "unknown dtype %d or epilogue %d", dt, epi);
    // The kernel's schedule arithmetic is 32-bit: work units (tiles x slices)
    // must number fewer than 2^31.
    if (cfg.bm > 0 && cfg.bn > 0 && cfg.split_k > 0 &&
        cdiv(cfg.swap_ab ? N : M, cfg.bm) * cdiv(cfg.swap_ab ? M : N, cfg.bn) * cfg.split_k >= ((int64_t)1 << 31))
        return set_error(GEMM_ERR_UNSUPPORTED, "the problem needs 2^31 or more work units with this configuration");
    if (dt == GEMM_MXFP8_E4M3 && std::max(mx_row_atoms(M), mx_row_atoms(N)) * mx_k_atoms(K) >= ((int64_t)1 << 31))
        return set_error(GEMM_ERR_UNSUPPORTED, "block-scaled FP8: the packed scales exceed 2^31 atoms");
    const int reason = check_config(M, N, K, dt, epi, cfg, dev);
    if (reason == GEMM_REASON_ALIGN)
        return set_error(GEMM_ERR_MISALIGNED, "K=%lld / N=%lld: %s", (long long)K, (long long)N, reason_text(reason));
    if (reason != GEMM_FEASIBLE)
        return set_error(GEMM_ERR_INFEASIBLE, "config %dx%dx%d s%d r%d g%d k%d c%d sw%d: %s", cfg.bm, cfg.bn, cfg.bk,
                         cfg.stages, cfg.raster, cfg.group, cfg.split_k, cfg.cta_group, cfg.swap_ab,
                         reason_text(reason));
    gemm_plan_s *p = new gemm_plan_s();
    p->M = M;
    p->N = N;
    p->K = K;
    p->dt = dt;
    p->epi = epi;
    p->cfg = cfg;
    p->dev = dev;
    cudaGetDevice(&p->device);
    p->L = layout_of(cfg, dt);
    const int route = g_b_route.load();
    p->b_kmajor = route == 1 || (route == 0 && !b_in_place(dt, N));
    // The kernel's bias/activation code; the residual is a run argument.
    p->kp = kernel_params_of(M, N, K, dt, act_code(epi), cfg, p->b_kmajor);
    KernelParams &k = p->kp;
    // One tensor copy per operand and stage where a stage spans several
    // 128-byte spans of an operand whose contiguous extent is a whole number of
    // spans (so that the 3-D view stays inside the matrix): the TMA unit takes
    // about as long over a copy whatever its size.  MMA-A's contiguous extent is
    // K (K-major) or N (B in place, swapped); MMA-B's K or N likewise.
    if (g_span3d.load()) {
        const int span = span_elems(dt);
        const int cta_rows = k.pair ? 128 : cfg.bm, cta_bcols = k.pair ? cfg.bn / 2 : cfg.bn;
        const int a_loads = k.a_mn_major ? cta_rows / span : cfg.bk / span;
        const int b_loads = k.b_mn_major ? cta_bcols / span : cfg.bk / span;
        k.a_span3d = a_loads > 1 && (k.a_mn_major ? N : K) % span == 0 ? 1 : 0;
        k.b_span3d = b_loads > 1 && (k.b_mn_major ? N : K) % span == 0 ? 1 : 0;
    }
    p->tiles = (int64_t)k.tiles_m * k.tiles_n;
    p->grid = (int)std::min<int64_t>(k.num_units, dev.sm_count);
    // One wave of split-K units: the slices of a tile finalise it share by
    // share, each owner its own unless a peer is late (no slice ever waits for
    // one that may not be resident).  The fix-up stages partials in the idle
    // pipeline ring: it needs 8 warps x 4 KB of it.
    const bool ring_room = p->L.off_staging >= 8u * 4096u;
    k.coop_fixup = (cfg.split_k > 1 && k.num_units <= dev.sm_count && !k.pair && ring_room) ? 1 : 0;
    // Or the slices of a tile form a cluster and reduce through distributed
    // shared memory (decided below, once the shared-memory limit is set).  Only
    // for one wave: past it, one CTA per unit loses the persistent schedule's
    // overlap, which costs more than the global exchange it replaces.
    const bool want_cluster = g_split_route.load() == 0 && k.num_units * (k.pair ? 2 : 1) <= dev.sm_count &&
                              cluster_reduce_fits(cfg, dt);
    // Ask for more than half of the SM's shared memory so that no two CTAs of
    // this kernel share an SM (each may hold up to 512 TMEM columns).
    const int64_t one_per_sm = dev.smem_per_block / 2 + 1024;
    p->smem_request = (int)std::min<int64_t>(dev.smem_per_block, std::max<int64_t>(p->L.smem_total, one_per_sm));

    // Split-K counters: one per exchange tile (a pair's tile is two, one per CTA).
    const int64_t n_counters = p->tiles * (k.pair ? 2 : 1);
    cudaError_t e = cudaMalloc(&p->aux, (size_t)(1 + n_counters) * sizeof(int32_t));
    if (e != cudaSuccess) {
        delete p;
        return cuda_err(e, "cudaMalloc(plan status/counters)");
    }
    e = cudaMemset(p->aux, 0, (size_t)(1 + n_counters) * sizeof(int32_t));
    if (e != cudaSuccess) {
        cudaFree(p->aux);
        delete p;
        return cuda_err(e, "cudaMemset(plan status/counters)");
    }
    k.status = p->aux;
    k.counters = p->aux + 1;
    p->n_counters = n_counters;
    if (cfg.split_k > 1) {
        const size_t n_counts = (size_t)n_counters * (size_t)cfg.split_k;   // one per share of a tile
        e = cudaMalloc(&p->epochs, n_counts * sizeof(uint64_t));
        if (e == cudaSuccess) e = cudaMemset(p->epochs, 0, n_counts * sizeof(uint64_t));
        if (e != cudaSuccess) {
            cudaFree(p->epochs);
            cudaFree(p->aux);
            delete p;
            return cuda_err(e, "cudaMalloc(split-K epochs)");
        }
    }
    k.epochs = p->epochs;
    if (cfg.split_k > 1) {
        if (shared_ws) {
            p->workspace = shared_ws;
        } else {
            const size_t bytes = (size_t)p->tiles * cfg.split_k * cfg.bm * cfg.bn * sizeof(float);
            e = cudaMalloc(&p->workspace, bytes);
            if (e != cudaSuccess) {
                cudaFree(p->aux);
                cudaFree(p->epochs);
                delete p;
                return cuda_err(e, "cudaMalloc(split-K workspace)");
            }
            p->owns_workspace = true;
        }
    }
    k.workspace = p->workspace;
    if (p->b_kmajor && K > 0 && N > 0) {
        e = cudaMalloc(&p->bt, (size_t)K * (size_t)N * elt_bytes(dt));
        if (e != cudaSuccess) {
            destroy_plan(p);
            return cuda_err(e, "cudaMalloc(K-major copy of B)");
        }
    }
    rc = configure_smem_limit(dt, dev.smem_per_block);
    if (rc) {
        destroy_plan(p);
        return rc;
    }
    if (k.pair) {
        // Pairs that fit at once: the persistent grid, and whether the split-K
        // units make one wave (one unit per pair; the slices then finalise
        // share by share, which needs no guarantee that they are resident
        // together).
        int pairs = 0;
        e = max_active_clusters(dt, k.a_mn_major, k.b_mn_major, 2, 2, p->smem_request, &pairs);
        if (e != cudaSuccess || pairs < 1) {
            cudaGetLastError();
            destroy_plan(p);
            return set_error(GEMM_ERR_INFEASIBLE, "no CTA pair of this configuration fits on the device");
        }
        p->grid = 2 * (int)std::min<int64_t>(k.num_units, pairs);
        k.coop_fixup = (cfg.split_k > 1 && k.num_units <= pairs && ring_room) ? 1 : 0;
    }
    if (want_cluster) {
        // Where shared memory allows, the partials get an area of their own past
        // the barriers (base + off_bar + 1 KB; the request's 1 KB alignment slack
        // stays), so the slices push without waiting for the owner's ring.
        const int64_t with_recv = (int64_t)p->L.smem_total + cluster_recv_bytes(cfg);
        const bool own_area = with_recv <= dev.smem_per_block;
        const int request = own_area ? (int)std::max<int64_t>(p->smem_request, with_recv) : p->smem_request;
        const int cg = k.pair ? 2 : 1;
        int clusters = 0;
        e = max_active_clusters(dt, k.a_mn_major, k.b_mn_major, cg, cfg.split_k * cg, request, &clusters);
        if (e != cudaSuccess) {
            cudaGetLastError();
            clusters = 0;
        }
        // Every cluster (one tile's S slices) resident at once: a cluster must
        // fit in one GPC, so large ones pack fewer than the SM count suggests
        // (8-CTA clusters of CTA pairs on 1000x1000x8192 ran in two waves, 45
        // against 24 us on the cooperative route).
        if (clusters > 0 && (int64_t)clusters * cfg.split_k >= k.num_units) {
            k.cluster_k = cfg.split_k;
            k.coop_fixup = 0;
            p->grid = (int)k.num_units * cg;  // one unit per CTA (per pair)
            if (own_area) {
                k.off_recv = p->L.off_bar + 1024u;
                p->smem_request = request;
            }
        }
    }
    *out = p;
    return GEMM_OK;
}

static size_t split_ws_bytes(int64_t M, int64_t N, const gemm_config &c)
{
    if (c.split_k <= 1) return 0;
    const int64_t rows = c.swap_ab ? N : M, cols = c.swap_ab ? M : N;
    return (size_t)(cdiv(rows, c.bm) * cdiv(cols, c.bn)) * c.split_k * c.bm * c.bn * sizeof(float);
}

void destroy_plan(gemm_plan_t p)
{
    if (!p) return;
    cudaFree(p->bt);
    if (p->owns_workspace) cudaFree(p->workspace);
    cudaFree(p->aux);
    cudaFree(p->epochs);
    cudaFree(p->hA);
    cudaFree(p->hB);
    cudaFree(p->hBias);
    cudaFree(p->hC);
    destroy_plan(p->twin);
    if (p->side) cudaStreamDestroy(p->side);
    delete p;
}

// A packed MX scale array as a 3-D tensor of 32-bit words: [row atoms][K atoms]
// [128 words] (one 512-byte atom per 128 words).  The box takes a stage's whole
// run for one operand in a single copy: bk/128 K atoms of each of the tile's
// `box_atoms` row atoms (each copy costs the TMA unit about as much as a data
// stage's, whatever its size, so one copy per operand and stage, not per atom).
static int encode_scales(CUtensorMap *m, const void *ptr, int64_t row_atoms, int64_t k_atoms, uint32_t ka,
                         uint32_t box_atoms)
{
    if (!encoder_ready()) return set_error(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[3] = {128, (cuuint64_t)k_atoms, (cuuint64_t)row_atoms};
    const cuuint64_t strides[2] = {512, (cuuint64_t)k_atoms * 512};
    const cuuint32_t box[3] = {128, ka, box_atoms};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return set_error(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for the MX scales [%lld x %lld atoms]",
                         (int)r, (long long)row_atoms, (long long)k_atoms);
    return GEMM_OK;
}

static int get_descs(gemm_plan_t p, const void *A, const void *B, void *C, const void *SA, const void *SB,
                     const DescEntry **out)
{
    for (const DescEntry &d : p->descs)
        if (d.valid && d.a == A && d.b == B && d.c == C && d.sa == SA && d.sb == SB) {
            *out = &d;
            return GEMM_OK;
        }
    DescEntry &d = p->descs[p->next_desc];
    p->next_desc = (p->next_desc + 1) % (int)p->descs.size();
    d.valid = false;
    const int dt = p->dt;
    const int span = span_elems(dt);
    const gemm_config &c = p->cfg;
    int rc = GEMM_OK;
    memset(&d.ma, 0, sizeof(d.ma));
    memset(&d.mb, 0, sizeof(d.mb));
    if (p->K > 0) {
        // A: [M, K] K-major, box [MMA extent x one span of K].
        // B: [K, N] read MN-major (box [bk x one span of N]) or its transposed
        //    copy [N, K] read K-major (box [MMA extent x one span of K]).
        // A's and B's extents per CTA (a CTA pair loads 128 rows of A and half
        // of B's columns in each CTA).
        const bool pair = c.cta_group == 2;
        const uint32_t a_rows = c.swap_ab ? c.bn : (pair ? 128u : (uint32_t)c.bm);
        const uint32_t b_rows = c.swap_ab ? c.bm : (pair ? (uint32_t)c.bn / 2 : (uint32_t)c.bn);
        CUtensorMap *am = c.swap_ab ? &d.mb : &d.ma;
        CUtensorMap *bm = c.swap_ab ? &d.ma : &d.mb;
        // Whether each matrix is read in spans (one copy per stage): A is
        // MMA-A unless swapped, B the other one.
        const bool a_spans = (c.swap_ab ? p->kp.b_span3d : p->kp.a_span3d) != 0;
        const bool b_spans = (c.swap_ab ? p->kp.a_span3d : p->kp.b_span3d) != 0;
        const uint32_t k_spans = (uint32_t)c.bk / (uint32_t)span;
        if (a_spans)
            rc = encode_spans(am, dt, A, p->K, p->M, span, a_rows, k_spans);
        else
            rc = encode_2d(am, dt, A, p->K, p->M, span, a_rows, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
        if (!rc) {
            if (p->b_kmajor && b_spans)
                rc = encode_spans(bm, dt, p->bt, p->K, p->N, span, b_rows, k_spans);
            else if (p->b_kmajor)
                rc = encode_2d(bm, dt, p->bt, p->K, p->N, span, b_rows, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
            else if (b_spans)
                rc = encode_spans(bm, dt, B, p->N, p->K, span, c.bk, b_rows / (uint32_t)span);
            else
                rc = encode_2d(bm, dt, B, p->N, p->K, span, c.bk, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
        }
    }
    if (!rc) {
        const int odt = is_fp8(dt) ? GEMM_BF16 : dt;   // C's type
        // A gated epilogue writes C of half the fused width.
        const uint64_t c_cols = is_glu(p->epi) ? (uint64_t)p->N / 2 : (uint64_t)p->N;
        if (!c.swap_ab)
            rc = encode_2d(&d.mc, odt, C, c_cols, p->M, 32, 32,
                           odt == GEMM_BF16 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_NONE);
        else
            rc = encode_2d(&d.mc, odt, C, p->N, p->M, 32, 16, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_NONE);
    }
    memset(&d.msa, 0, sizeof(d.msa));
    memset(&d.msb, 0, sizeof(d.msb));
    if (!rc && dt == GEMM_MXFP8_E4M3 && p->K > 0) {
        // Row atoms per copy: the MMA-A side of a tile (one per CTA of a pair,
        // else bm/128) and the MMA-B side (bn/128, at least one); swapped, B's
        // scales feed MMA-A and A's MMA-B.
        const uint32_t ka = (uint32_t)c.bk / 128u;
        const uint32_t na = c.cta_group == 2 ? 1u : (uint32_t)c.bm / 128u;
        const uint32_t nb = (uint32_t)std::max(1, c.bn / 128);
        rc = encode_scales(&d.msa, SA, mx_row_atoms(p->M), mx_k_atoms(p->K), ka, c.swap_ab ? nb : na);
        if (!rc) rc = encode_scales(&d.msb, SB, mx_row_atoms(p->N), mx_k_atoms(p->K), ka, c.swap_ab ? na : nb);
    }
    if (rc) return rc;
    d.a = A;
    d.b = B;
    d.c = C;
    d.sa = SA;
    d.sb = SB;
    d.valid = true;
    *out = &d;
    return GEMM_OK;
}

static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
static int read_status(gemm_plan_t p);

int run_plan_mx(gemm_plan_t p, const void *A, const void *SA, const void *B, const void *SB, const void *bias,
                const void *R, void *C, cudaStream_t stream)
{
    if (!p) return set_error(GEMM_ERR_INVALID_ARG, "null plan");
    const bool mx = p->dt == GEMM_MXFP8_E4M3;
    if (mx && p->K > 0 && (!SA || !SB))
        return set_error(GEMM_ERR_INVALID_ARG, "a block-scaled FP8 plan runs through gemm_run_mx, with both scales");
    if (!mx && (SA || SB)) return set_error(GEMM_ERR_INVALID_ARG, "scales given to a plan that is not block-scaled");
    if (mx && p->K > 0 && (!aligned16(SA) || !aligned16(SB)))
        return set_error(GEMM_ERR_MISALIGNED, "SA and SB must be 16-byte aligned");
    if (has_residual(p->epi) && !R)
        return set_error(GEMM_ERR_INVALID_ARG, "the residual epilogue needs R (gemm_run_ex)");
    if (!has_residual(p->epi) && R)
        return set_error(GEMM_ERR_INVALID_ARG, "R given to a plan whose epilogue has no residual");
    if (p->M == 0 || p->N == 0) return GEMM_OK;
    if (!C || (p->K > 0 && (!A || !B))) return set_error(GEMM_ERR_INVALID_ARG, "null A, B or C");
    if (p->epi != GEMM_EPI_NONE && !bias) return set_error(GEMM_ERR_INVALID_ARG, "bias is required by the epilogue");
    if ((p->K > 0 && (!aligned16(A) || !aligned16(B))) || !aligned16(C) ||
        (p->epi != GEMM_EPI_NONE && !aligned16(bias)) || (R && !aligned16(R)))
        return set_error(GEMM_ERR_MISALIGNED, "A, B, C, bias and R must be 16-byte aligned");
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev != p->device)
        return set_error(GEMM_ERR_INVALID_ARG, "plan was made on device %d, current device is %d", p->device, dev);
    const DescEntry *d = nullptr;
    int rc = get_descs(p, A, B, C, SA, SB, &d);
    if (rc) return rc;
    if (p->b_kmajor && p->K > 0) {
        cudaError_t te = launch_transpose(B, p->bt, p->K, p->N, elt_bytes(p->dt), stream);
        if (te != cudaSuccess) return cuda_err(te, "transpose launch");
    }
    KernelParams kp = p->kp;
    kp.bias = p->epi != GEMM_EPI_NONE ? bias : nullptr;
    kp.residual = R;
    kp.timeout_ns = g_timeout_ns.load();
    kp.debug_stall = g_debug_stall.load();
    kp.share_poll_cycles = g_share_poll.load();
    // Declared operands map to the kernel's MMA-A (bit 0) and MMA-B (bit 1);
    // swapped, MMA-A is B.  A K-major copy of B is written by the kernel just
    // before, so B then always waits.
    {
        const int32_t ua = p->independent & GEMM_OPERAND_A;
        const int32_t ub = p->b_kmajor ? 0 : (p->independent & GEMM_OPERAND_B);
        const int32_t ka = p->cfg.swap_ab ? ub : ua, kb = p->cfg.swap_ab ? ua : ub;
        kp.early_mask = (ka ? 1 : 0) | (kb ? 2 : 0);
    }
    cudaError_t e = launch_gemm(p->dt, d->ma, d->mb, d->mc, mx ? &d->msa : nullptr, mx ? &d->msb : nullptr, kp, p->grid,
                                p->smem_request, stream);
    if (e != cudaSuccess) return cuda_err(e, "kernel launch");
    if (g_check.load()) {
        e = cudaStreamSynchronize(stream);
        if (e != cudaSuccess) return cuda_err(e, "cudaStreamSynchronize (checked run)");
        return read_status(p);
    }
    return GEMM_OK;
}

int run_plan_ex(gemm_plan_t p, const void *A, const void *B, const void *bias, const void *R, void *C,
                cudaStream_t stream)
{
    return run_plan_mx(p, A, nullptr, B, nullptr, bias, R, C, stream);
}

int run_plan(gemm_plan_t p, const void *A, const void *B, const void *bias, void *C, cudaStream_t stream)
{
    return run_plan_ex(p, A, B, bias, nullptr, C, stream);
}

int mx_pack_scales(const void *scales, int64_t rows, int64_t K, int b_side, void *packed, cudaStream_t stream)
{
    if (rows < 0 || K < 0) return set_error(GEMM_ERR_INVALID_ARG, "negative extent");
    if (b_side != 0 && b_side != 1) return set_error(GEMM_ERR_INVALID_ARG, "b_side must be 0 (A) or 1 (B)");
    if (rows == 0 || K == 0) return GEMM_OK;
    if (!scales || !packed) return set_error(GEMM_ERR_INVALID_ARG, "null scales or packed buffer");
    cudaError_t e = launch_mx_pack(static_cast<const uint8_t *>(scales), rows, K, b_side,
                                   static_cast<uint8_t *>(packed), stream);
    if (e != cudaSuccess) return cuda_err(e, "MX scale packing launch");
    return GEMM_OK;
}

int plan_set_independent_operands(gemm_plan_t p, int32_t mask)
{
    if (!p) return set_error(GEMM_ERR_INVALID_ARG, "null plan");
    if (mask & ~(GEMM_OPERAND_A | GEMM_OPERAND_B)) return set_error(GEMM_ERR_INVALID_ARG, "unknown operand bits");
    p->independent = mask;
    return GEMM_OK;
}

int plan_set_scale(gemm_plan_t p, float alpha)
{
    if (!p) return set_error(GEMM_ERR_INVALID_ARG, "null plan");
    if (!(fabsf(alpha) <= 3.402823466e38f)) return set_error(GEMM_ERR_INVALID_ARG, "the scale must be finite");
    p->kp.alpha = alpha;
    return GEMM_OK;
}

int plan_launch_info(gemm_plan_t p, gemm_launch_info *out)
{
    const KernelParams &k = p->kp;
    memset(out, 0, sizeof(*out));
    out->grid = p->grid;
    out->block = kThreadsPerCta;
    out->smem_bytes = p->smem_request;
    out->cluster = k.cluster_k > 1 ? k.cluster_k * (k.pair ? 2 : 1) : k.pair ? 2 : 1;
    out->splitk_route = p->cfg.split_k <= 1 ? 0 : k.cluster_k > 1 ? 3 : k.coop_fixup ? 2 : 1;
    out->b_transposed = p->b_kmajor ? 1 : 0;
    out->units = k.num_units;
    out->tiles = (int32_t)p->tiles;
    out->span_copies = (k.a_span3d ? 1 : 0) | (k.b_span3d ? 2 : 0);
    return GEMM_OK;
}

int plan_config(gemm_plan_t p, gemm_config *out)
{
    if (!p || !out) return set_error(GEMM_ERR_INVALID_ARG, "null plan or output");
    *out = p->cfg;
    return GEMM_OK;
}

int plan_status(gemm_plan_t p)
{
    if (!p) return set_error(GEMM_ERR_INVALID_ARG, "null plan");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_err(e, "cudaDeviceSynchronize");
    return read_status(p);
}

// The plan's device status word, after its work has finished: GEMM_OK, or
// GEMM_ERR_TIMEOUT with the word and the split-K counters reset.
static int read_status(gemm_plan_t p)
{
    int32_t st = 0;
    cudaError_t e = cudaMemcpy(&st, p->aux, sizeof(st), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_err(e, "reading the status word");
    if (st != 0) {
        // An early return may leave counts part-way: start them afresh.
        cudaMemset(p->aux, 0, (size_t)(1 + p->n_counters) * sizeof(int32_t));
        if (p->epochs) cudaMemset(p->epochs, 0, (size_t)p->n_counters * p->cfg.split_k * sizeof(uint64_t));
        return set_error(GEMM_ERR_TIMEOUT, "a device wait expired (site %d); the kernel returned early", st);
    }
    return GEMM_OK;
}

// Plan-owned device buffers for runs from host memory (allocated on first use).
static int host_run_buffers(gemm_plan_t p)
{
    if (p->hC) return GEMM_OK;
    const size_t e = (size_t)elt_bytes(p->dt), eo = (size_t)out_elt_bytes(p->dt);
    const size_t nA = (size_t)p->M * p->K * e, nB = (size_t)p->K * p->N * e, nBias = (size_t)p->N * eo,
                 nC = (size_t)p->M * (is_glu(p->epi) ? p->N / 2 : p->N) * eo;
    cudaError_t err;
    if ((nA && (err = cudaMalloc(&p->hA, nA)) != cudaSuccess) || (nB && (err = cudaMalloc(&p->hB, nB)) != cudaSuccess) ||
        (err = cudaMalloc(&p->hBias, nBias)) != cudaSuccess || (err = cudaMalloc(&p->hC, nC)) != cudaSuccess)
        return cuda_err(err, "cudaMalloc(host-run buffers)");
    return GEMM_OK;
}

// Copies one GEMM's inputs in, runs it, and queues the copy of C back, all on `stream`.
static int host_run_enqueue(gemm_plan_t p, const void *A, const void *B, const void *bias, void *C,
                            cudaStream_t stream)
{
    const size_t e = (size_t)elt_bytes(p->dt), eo = (size_t)out_elt_bytes(p->dt);
    const size_t nA = (size_t)p->M * p->K * e, nB = (size_t)p->K * p->N * e, nBias = (size_t)p->N * eo,
                 nC = (size_t)p->M * (is_glu(p->epi) ? p->N / 2 : p->N) * eo;
    const bool has_bias = p->epi != GEMM_EPI_NONE;
    if (has_bias && !bias) return set_error(GEMM_ERR_INVALID_ARG, "bias is required by the epilogue");
    if (!C || (p->K > 0 && (!A || !B))) return set_error(GEMM_ERR_INVALID_ARG, "null A, B or C");
    cudaError_t err;
    if (nA && (err = cudaMemcpyAsync(p->hA, A, nA, cudaMemcpyHostToDevice, stream)) != cudaSuccess)
        return cuda_err(err, "copy A to device");
    if (nB && (err = cudaMemcpyAsync(p->hB, B, nB, cudaMemcpyHostToDevice, stream)) != cudaSuccess)
        return cuda_err(err, "copy B to device");
    if (has_bias && (err = cudaMemcpyAsync(p->hBias, bias, nBias, cudaMemcpyHostToDevice, stream)) != cudaSuccess)
        return cuda_err(err, "copy bias to device");
    int rc = run_plan(p, p->hA, p->hB, has_bias ? p->hBias : nullptr, p->hC, stream);
    if (rc) return rc;
    if ((err = cudaMemcpyAsync(C, p->hC, nC, cudaMemcpyDeviceToHost, stream)) != cudaSuccess)
        return cuda_err(err, "copy C to host");
    return GEMM_OK;
}

int run_host(gemm_plan_t p, const void *A, const void *B, const void *bias, void *C, cudaStream_t stream)
{
    if (!p) return set_error(GEMM_ERR_INVALID_ARG, "null plan");
    if (p->M == 0 || p->N == 0) return GEMM_OK;
    int rc = host_run_buffers(p);
    if (!rc) rc = host_run_enqueue(p, A, B, bias, C, stream);
    if (rc) return rc;
    cudaError_t err = cudaStreamSynchronize(stream);
    if (err != cudaSuccess) return cuda_err(err, "cudaStreamSynchronize");
    return GEMM_OK;
}

// n GEMMs of the plan's shape from host buffers, pipelined: GEMM i runs on
// `stream` when i is even and on the plan's second stream (with a second plan
// of the same configuration, whose split-K state is its own) when i is odd, so
// the copies of one GEMM overlap the kernel of the other.  Returns once every
// C is in host memory, with both plans' device status words read.
int run_host_many(gemm_plan_t p, int n, const void *const *A, const void *const *B, const void *const *bias,
                  void *const *C, cudaStream_t stream)
{
    if (!p) return set_error(GEMM_ERR_INVALID_ARG, "null plan");
    if (n < 0 || (n > 0 && (!A || !B || !C))) return set_error(GEMM_ERR_INVALID_ARG, "bad GEMM count or null arrays");
    if (p->epi != GEMM_EPI_NONE && n > 0 && !bias) return set_error(GEMM_ERR_INVALID_ARG, "null bias array");
    if (n == 0 || p->M == 0 || p->N == 0) return GEMM_OK;
    int rc = host_run_buffers(p);
    if (rc) return rc;
    cudaError_t err;
    if (n > 1 && !p->twin) {
        rc = make_plan(p->M, p->N, p->K, p->dt, p->epi, p->cfg, p->dev, nullptr, &p->twin);
        if (rc) return rc;
        if ((rc = host_run_buffers(p->twin))) return rc;
    }
    if (n > 1 && !p->side && (err = cudaStreamCreateWithFlags(&p->side, cudaStreamNonBlocking)) != cudaSuccess)
        return cuda_err(err, "cudaStreamCreate");
    if (p->twin) {
        p->twin->kp.alpha = p->kp.alpha;
        p->twin->independent = p->independent;
    }
    cudaEvent_t ev = nullptr;
    if (n > 1) {
        // the second stream starts after the work queued on the caller's stream
        if ((err = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess)
            return cuda_err(err, "cudaEventCreate");
        cudaEventRecord(ev, stream);
        cudaStreamWaitEvent(p->side, ev, 0);
    }
    for (int i = 0; i < n && !rc; ++i) {
        const bool odd = (i & 1) != 0;
        rc = host_run_enqueue(odd ? p->twin : p, A[i], B[i], bias ? bias[i] : nullptr, C[i], odd ? p->side : stream);
    }
    cudaError_t e1 = cudaStreamSynchronize(stream);
    cudaError_t e2 = p->side ? cudaStreamSynchronize(p->side) : cudaSuccess;
    if (ev) cudaEventDestroy(ev);
    if (rc) return rc;
    if (e1 != cudaSuccess) return cuda_err(e1, "cudaStreamSynchronize");
    if (e2 != cudaSuccess) return cuda_err(e2, "cudaStreamSynchronize (second stream)");
    rc = read_status(p);
    if (!rc && p->twin && n > 1) rc = read_status(p->twin);
    return rc;
}

// ---------------------------------------------------------------------------
// Tuner
// ---------------------------------------------------------------------------

struct TuneBuffers {
    std::vector<void *> A, B, bias, C, SA, SB;   // SA, SB: packed MX scales (block-scaled FP8 only)
    float *ws = nullptr;
    ~TuneBuffers()
    {
        for (auto *v : {&A, &B, &bias, &C, &SA, &SB})
            for (void *p : *v) cudaFree(p);
        cudaFree(ws);
    }
};

static double median_of(std::vector<double> v)
{
    std::sort(v.begin(), v.end());
    const size_t n = v.size();
    if (n == 0) return -1.0;
    return n % 2 ? v[n / 2] : 0.5 * (v[n / 2 - 1] + v[n / 2]);
}

static int env_int(const char *name, int dflt)
{
    const char *v = getenv(name);
    if (!v || !*v) return dflt;
    return atoi(v);
}

int tune(int64_t M, int64_t N, int64_t K, int dt, int epi, int mode, int topk, uint64_t seed,
         std::vector<gemm_tune_row> &rows, gemm_rank_stats &stats, gemm_config *winner,
         const gemm_config *list, int nlist, const TuneInputs *user)
{
    const auto t_start = std::chrono::steady_clock::now();
    memset(&stats, 0, sizeof(stats));
    stats.fixed_us = -1.0;
    rows.clear();
    int rc = check_extents(M, N, K);
    if (rc) return rc;
    if (!valid_enums(dt, epi)) return set_error(GEMM_ERR_INVALID_ARG, "unknown dtype %d or epilogue %d", dt, epi);
    if ((rc = check_device_arch(nullptr))) return rc;
    gemm_device_params dev;
    if ((rc = query_params(&dev))) return rc;
    // Candidates: the generator's, or the feasible members of a given list (a
    // shipped configuration set), every one of which is timed.
    std::vector<gemm_config> cands;
    if (list) {
        for (int i = 0; i < nlist; ++i) {
            if (check_config(M, N, K, dt, epi, list[i], dev) != GEMM_FEASIBLE) continue;
            bool dup = false;
            for (const gemm_config &c : cands) dup = dup || memcmp(&c, &list[i], sizeof(c)) == 0;
            if (!dup) cands.push_back(list[i]);
        }
        if (cands.empty())
            return set_error(GEMM_ERR_UNSUPPORTED, "no configuration of the list runs M=%lld N=%lld K=%lld",
                             (long long)M, (long long)N, (long long)K);
        mode = GEMM_SEARCH_EXHAUSTIVE;
    } else {
        cands = enumerate(M, N, K, dt, epi, dev);
    }
    if (cands.empty()) {
        const int reason = check_config(M, N, K, dt, epi, fixed_config(dt, dev), dev);
        if (reason == GEMM_REASON_ALIGN) return set_error(GEMM_ERR_MISALIGNED, "%s", reason_text(reason));
        return set_error(GEMM_ERR_UNSUPPORTED, "no feasible configuration for M=%lld N=%lld K=%lld", (long long)M,
                         (long long)N, (long long)K);
    }
    const gemm_config fixed = fixed_config(dt, dev);
    const int n = (int)cands.size();
    rows.resize(n);
    std::vector<double> pred(n);
    for (int i = 0; i < n; ++i) {
        memset(&rows[i], 0, sizeof(gemm_tune_row));
        rows[i].config = cands[i];
        pred[i] = predict(M, N, K, dt, epi, cands[i], dev).predicted_us;
        rows[i].predicted_us = pred[i];
        rows[i].measured_us = -1.0;
        rows[i].measured_min_us = -1.0;
        rows[i].measured_rank = -1;
    }
    std::vector<int> by_model(n);
    std::iota(by_model.begin(), by_model.end(), 0);
    std::stable_sort(by_model.begin(), by_model.end(), [&](int a, int b) { return pred[a] < pred[b]; });
    for (int r = 0; r < n; ++r) rows[by_model[r]].model_rank = r;
    auto same = [](const gemm_config &a, const gemm_config &b) { return memcmp(&a, &b, sizeof(a)) == 0; };
    int fixed_idx = -1;
    for (int i = 0; i < n; ++i)
        if (same(cands[i], fixed)) fixed_idx = i;

    // Which candidates to time ("Autotuning & cost models" §6): every one
    // (exhaustive), the model's top-k plus the fixed tile (model-guided), or k
    // drawn uniformly at random with a seeded splitmix64 stream (random-k).
    std::vector<int> meas;
    if (mode == GEMM_SEARCH_EXHAUSTIVE || topk <= 0 || topk >= n) {
        meas = by_model;
    } else if (mode == GEMM_SEARCH_RANDOM_K) {
        std::vector<int> pool(n);
        std::iota(pool.begin(), pool.end(), 0);
        uint64_t x = seed;
        for (int i = 0; i < topk; ++i) {   // partial Fisher-Yates shuffle
            x += 0x9E3779B97F4A7C15ull;
            uint64_t z = x;
            z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
            z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
            z ^= z >> 31;
            const int j = i + (int)(z % (uint64_t)(n - i));
            std::swap(pool[i], pool[j]);
        }
        meas.assign(pool.begin(), pool.begin() + topk);
    } else {
        meas.assign(by_model.begin(), by_model.begin() + topk);
        if (fixed_idx >= 0 && std::find(meas.begin(), meas.end(), fixed_idx) == meas.end()) meas.push_back(fixed_idx);
    }
    const int nm = (int)meas.size();

    // Library-owned buffers, rotated so that shapes smaller than L2 are timed
    // from HBM like the real, larger working set.
    const size_t e = (size_t)elt_bytes(dt), eo = (size_t)out_elt_bytes(dt);
    const int odt = is_fp8(dt) ? GEMM_BF16 : dt;   // type of bias and C
    const bool mx = dt == GEMM_MXFP8_E4M3;
    const size_t bytes_sa = mx ? (size_t)std::max<int64_t>(mx_row_atoms(M) * mx_k_atoms(K) * kMxAtomBytes, 16) : 0,
                 bytes_sb = mx ? (size_t)std::max<int64_t>(mx_row_atoms(N) * mx_k_atoms(K) * kMxAtomBytes, 16) : 0;
    const size_t bytes_a = (size_t)std::max<int64_t>(M * K, 1) * e, bytes_b = (size_t)std::max<int64_t>(K * N, 1) * e,
                 bytes_bias = (size_t)std::max<int64_t>(N, 1) * eo, bytes_c = (size_t)std::max<int64_t>(M * N, 1) * eo;
    const size_t set_bytes = bytes_a + bytes_b + bytes_bias + bytes_c + bytes_sa + bytes_sb;
    int nsets = (int)std::min<int64_t>(8, std::max<int64_t>(1, cdiv(2 * dev.l2_bytes + (int64_t)set_bytes, set_bytes)));
    TuneBuffers buf;
    cudaStream_t stream = nullptr;
    cudaError_t err = cudaStreamCreateWithFlags(&stream, cudaStreamNonBlocking);
    if (err != cudaSuccess) return cuda_err(err, "cudaStreamCreate");
    struct StreamGuard {
        cudaStream_t s;
        ~StreamGuard() { cudaStreamDestroy(s); }
    } sg{stream};
    // Synthetic operands with the workloads' spread (standard deviation
    // 1/sqrt(K), "Tile Selection", "Measurement, and what it must control":
    // tuning inputs must resemble the real ones in distribution), or copies of
    // the caller's own operands.
    const int fill = g_tune_fill.load();
    const float sd = (float)(1.0 / sqrt((double)std::max<int64_t>(K, 1)));
    const float scale_ab = fill == 0 ? sd * (float)sqrt(3.0) : sd;
    if (user) {
        // the caller's operands are read on this private stream: finish what
        // the device has queued first (their producers may be on any stream)
        if ((err = cudaDeviceSynchronize()) != cudaSuccess) return cuda_err(err, "cudaDeviceSynchronize");
        const bool need_b = K > 0 && N > 0, need_a = K > 0 && M > 0;
        if ((need_a && !user->A) || (need_b && !user->B) || (epi != GEMM_EPI_NONE && !user->bias) ||
            (mx && K > 0 && (!user->SA || !user->SB)))
            return set_error(GEMM_ERR_INVALID_ARG, "tuning on given operands: A, B, bias (and MX scales) are needed");
    }
    for (int s = 0; s < nsets; ++s) {
        void *a = nullptr, *b = nullptr, *bb = nullptr, *c = nullptr;
        if ((err = cudaMalloc(&a, bytes_a)) != cudaSuccess) return cuda_err(err, "cudaMalloc(tuning A)");
        buf.A.push_back(a);
        if ((err = cudaMalloc(&b, bytes_b)) != cudaSuccess) return cuda_err(err, "cudaMalloc(tuning B)");
        buf.B.push_back(b);
        if ((err = cudaMalloc(&bb, bytes_bias)) != cudaSuccess) return cuda_err(err, "cudaMalloc(tuning bias)");
        buf.bias.push_back(bb);
        if ((err = cudaMalloc(&c, bytes_c)) != cudaSuccess) return cuda_err(err, "cudaMalloc(tuning C)");
        buf.C.push_back(c);
        if (user) {
            // Every set a copy of the caller's operands (distinct addresses, so
            // the rotation still keeps the timed GEMMs out of L2).
            if (M * K > 0) cudaMemcpyAsync(a, user->A, (size_t)(M * K) * e, cudaMemcpyDeviceToDevice, stream);
            if (K * N > 0) cudaMemcpyAsync(b, user->B, (size_t)(K * N) * e, cudaMemcpyDeviceToDevice, stream);
            if (epi != GEMM_EPI_NONE) cudaMemcpyAsync(bb, user->bias, (size_t)N * eo, cudaMemcpyDeviceToDevice, stream);
        } else {
            launch_fill_random(a, (int64_t)(bytes_a / e), dt, scale_ab, 0x1234u + 17u * s, fill, stream);
            launch_fill_random(b, (int64_t)(bytes_b / e), dt, scale_ab, 0x5678u + 17u * s, fill, stream);
            launch_fill_random(bb, (int64_t)(bytes_bias / eo), odt, 0.1f, 0x9ABCu + 17u * s, fill, stream);
        }
        if (mx) {
            // Packed scales: the caller's, or 2^0 (E8M0 127) for synthetic operands.
            void *sa = nullptr, *sb = nullptr;
            if ((err = cudaMalloc(&sa, bytes_sa)) != cudaSuccess) return cuda_err(err, "cudaMalloc(tuning SA)");
            buf.SA.push_back(sa);
            if ((err = cudaMalloc(&sb, bytes_sb)) != cudaSuccess) return cuda_err(err, "cudaMalloc(tuning SB)");
            buf.SB.push_back(sb);
            if (user && K > 0) {
                cudaMemcpyAsync(sa, user->SA, (size_t)(mx_row_atoms(M) * mx_k_atoms(K) * kMxAtomBytes),
                                cudaMemcpyDeviceToDevice, stream);
                cudaMemcpyAsync(sb, user->SB, (size_t)(mx_row_atoms(N) * mx_k_atoms(K) * kMxAtomBytes),
                                cudaMemcpyDeviceToDevice, stream);
            } else {
                cudaMemsetAsync(sa, 127, bytes_sa, stream);
                cudaMemsetAsync(sb, 127, bytes_sb, stream);
            }
        }
    }
    size_t ws_bytes = 0;
    for (int i : meas) ws_bytes = std::max(ws_bytes, split_ws_bytes(M, N, cands[i]));
    if (ws_bytes && (err = cudaMalloc(&buf.ws, ws_bytes)) != cudaSuccess) return cuda_err(err, "cudaMalloc(tuning workspace)");

    std::vector<gemm_plan_t> plans(nm, nullptr);
    struct PlanGuard {
        std::vector<gemm_plan_t> &v;
        ~PlanGuard()
        {
            for (auto p : v) destroy_plan(p);
        }
    } pg{plans};
    std::vector<int> status(nm, GEMM_OK);
    for (int j = 0; j < nm; ++j) {
        status[j] = make_plan(M, N, K, dt, epi, cands[meas[j]], dev, buf.ws, &plans[j]);
    }
    // (A residual epilogue is timed in place: R = C.)
    auto run_one = [&](int j, int set) {
        return run_plan_mx(plans[j], buf.A[set], mx ? buf.SA[set] : nullptr, buf.B[set], mx ? buf.SB[set] : nullptr,
                           epi != GEMM_EPI_NONE ? buf.bias[set] : nullptr, has_residual(epi) ? buf.C[set] : nullptr,
                           buf.C[set], stream);
    };
    // Warm-up and a first estimate of each candidate's time.
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    std::vector<int> reps(nm, 1);
    for (int j = 0; j < nm; ++j) {
        if (status[j]) continue;
        for (int w = 0; w < 2 && !status[j]; ++w) status[j] = run_one(j, w % nsets);
        if (status[j]) continue;
        cudaEventRecord(e0, stream);
        status[j] = run_one(j, 2 % nsets);
        cudaEventRecord(e1, stream);
        if ((err = cudaEventSynchronize(e1)) != cudaSuccess) {
            cudaEventDestroy(e0);
            cudaEventDestroy(e1);
            return cuda_err(err, "tuning warm-up");
        }
        if (!status[j]) status[j] = plan_status(plans[j]);
        float ms = 0;
        cudaEventElapsedTime(&ms, e0, e1);
        const double us = std::max(1.0, ms * 1000.0);
        reps[j] = (int)std::min(200.0, std::max(1.0, ceil(300.0 / us)));
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    // Interleaved rounds: every round times every candidate once, starting at a
    // different candidate, so clock drift is spread over all of them.
    const int rounds = std::max(1, env_int("GEMM_TUNE_ROUNDS", 5));
    std::vector<std::vector<double>> times(nm);
    std::vector<cudaEvent_t> ev(2 * nm);
    for (auto &x : ev) cudaEventCreate(&x);
    int set = 0;
    for (int r = 0; r < rounds; ++r) {
        for (int t = 0; t < nm; ++t) {
            const int j = (t + r) % nm;
            if (status[j]) continue;
            cudaEventRecord(ev[2 * j], stream);
            for (int q = 0; q < reps[j] && !status[j]; ++q) {
                status[j] = run_one(j, set);
                set = (set + 1) % nsets;
            }
            cudaEventRecord(ev[2 * j + 1], stream);
        }
        if ((err = cudaStreamSynchronize(stream)) != cudaSuccess) {
            for (auto &x : ev) cudaEventDestroy(x);
            return cuda_err(err, "tuning round");
        }
        for (int j = 0; j < nm; ++j) {
            if (status[j]) continue;
            float ms = 0;
            cudaEventElapsedTime(&ms, ev[2 * j], ev[2 * j + 1]);
            times[j].push_back(ms * 1000.0 / reps[j]);
        }
    }
    for (auto &x : ev) cudaEventDestroy(x);
    for (int j = 0; j < nm; ++j)
        if (!status[j]) status[j] = plan_status(plans[j]);

    std::vector<int> ok_idx;
    for (int j = 0; j < nm; ++j) {
        gemm_tune_row &row = rows[meas[j]];
        row.status = status[j];
        if (status[j] || times[j].empty()) continue;
        row.measured_us = median_of(times[j]);
        row.measured_min_us = *std::min_element(times[j].begin(), times[j].end());
        ok_idx.push_back(meas[j]);
    }
    if (ok_idx.empty()) return set_error(GEMM_ERR_CUDA, "no candidate could be timed");
    std::stable_sort(ok_idx.begin(), ok_idx.end(), [&](int a, int b) {
        if (rows[a].measured_us != rows[b].measured_us) return rows[a].measured_us < rows[b].measured_us;
        return rows[a].model_rank < rows[b].model_rank;
    });
    for (size_t r = 0; r < ok_idx.size(); ++r) rows[ok_idx[r]].measured_rank = (int)r;
    std::vector<double> pm, mm;
    for (int i : ok_idx) {
        pm.push_back(rows[i].predicted_us);
        mm.push_back(rows[i].measured_us);
    }
    if (pm.size() >= 2) stats = rank_agreement(pm.data(), mm.data(), (int)pm.size());
    stats.best_us = rows[ok_idx[0]].measured_us;
    stats.fixed_us = (fixed_idx >= 0 && rows[fixed_idx].measured_us > 0) ? rows[fixed_idx].measured_us : -1.0;
    stats.n_measured = (int)ok_idx.size();
    stats.n_candidates = n;
    if (winner) *winner = rows[ok_idx[0]].config;
    // Rows ordered by measured time, unmeasured rows last (by model rank).
    std::vector<gemm_tune_row> sorted;
    for (int i : ok_idx) sorted.push_back(rows[i]);
    std::vector<int> rest;
    for (int i = 0; i < n; ++i)
        if (rows[i].measured_rank < 0) rest.push_back(i);
    std::stable_sort(rest.begin(), rest.end(), [&](int a, int b) { return rows[a].model_rank < rows[b].model_rank; });
    for (int i : rest) sorted.push_back(rows[i]);
    rows.swap(sorted);
    stats.tune_seconds = std::chrono::duration<double>(std::chrono::steady_clock::now() - t_start).count();
    return GEMM_OK;
}

// ---------------------------------------------------------------------------
// Tune-once cache keyed by (M, N, K, dtype, epilogue, device name, SM count,
// library version)
// ---------------------------------------------------------------------------

static std::mutex g_cache_mu;
static std::map<std::string, gemm_config> g_cache;
static int64_t g_tunes = 0, g_hits = 0;

// Tuning database file ("Tile Selection": tuned results are "shipped with the
// artifact or stored in a tuning database that persists across deployments";
// "Autotuning & cost models" §5: AOT tuning log).  One text line per entry:
//   <key> TAB bm bn bk stages raster group split_k cta_group swap_ab
// with <key> = M|N|K|dtype|epilogue|device name|SM count|library version, so an
// entry only ever serves the device and library version that produced it.
static bool parse_db_line(const std::string &line, std::string &key, gemm_config &c)
{
    const size_t tab = line.find('\t');
    if (tab == std::string::npos || tab == 0) return false;
    key = line.substr(0, tab);
    int v[9];
    if (sscanf(line.c_str() + tab + 1, "%d %d %d %d %d %d %d %d %d", &v[0], &v[1], &v[2], &v[3], &v[4], &v[5], &v[6],
               &v[7], &v[8]) != 9)
        return false;
    c = gemm_config{v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7], v[8]};
    return true;
}

static std::string db_line(const std::string &key, const gemm_config &c)
{
    char buf[128];
    snprintf(buf, sizeof(buf), "\t%d %d %d %d %d %d %d %d %d\n", c.bm, c.bn, c.bk, c.stages, c.raster, c.group,
             c.split_k, c.cta_group, c.swap_ab);
    return key + buf;
}

// Requires g_cache_mu held.
static int load_db_locked(const char *path, int64_t *n)
{
    FILE *f = fopen(path, "r");
    if (!f) return set_error(GEMM_ERR_INVALID_ARG, "cannot open tuning database '%s'", path);
    int64_t count = 0;
    char buf[1024];
    while (fgets(buf, sizeof(buf), f)) {
        std::string line(buf), key;
        while (!line.empty() && (line.back() == '\n' || line.back() == '\r')) line.pop_back();
        gemm_config c;
        if (line.empty() || line[0] == '#' || !parse_db_line(line, key, c)) continue;
        g_cache[key] = c;
        ++count;
    }
    fclose(f);
    if (n) *n = count;
    return GEMM_OK;
}

int cache_save(const char *path, int64_t *n)
{
    if (!path) return set_error(GEMM_ERR_INVALID_ARG, "null path");
    std::lock_guard<std::mutex> lk(g_cache_mu);
    const std::string tmp = std::string(path) + ".tmp";
    FILE *f = fopen(tmp.c_str(), "w");
    if (!f) return set_error(GEMM_ERR_INVALID_ARG, "cannot write tuning database '%s'", path);
    fprintf(f, "# tuning database of %s: key TAB bm bn bk stages raster group split_k cta_group swap_ab\n",
            GEMM_LIB_VERSION);
    for (const auto &kv : g_cache) fputs(db_line(kv.first, kv.second).c_str(), f);
    const bool ok = fclose(f) == 0 && rename(tmp.c_str(), path) == 0;
    if (!ok) return set_error(GEMM_ERR_INVALID_ARG, "cannot replace tuning database '%s'", path);
    if (n) *n = (int64_t)g_cache.size();
    return GEMM_OK;
}

int cache_load(const char *path, int64_t *n)
{
    if (!path) return set_error(GEMM_ERR_INVALID_ARG, "null path");
    std::lock_guard<std::mutex> lk(g_cache_mu);
    return load_db_locked(path, n);
}

// GEMM_TUNING_DB=<path>: loaded on the first tuned plan, appended to on every
// new winner (just-in-time tuning that persists).
static const char *db_path()
{
    const char *p = getenv("GEMM_TUNING_DB");
    return (p && *p) ? p : nullptr;
}

static std::string cache_key(int64_t M, int64_t N, int64_t K, int dt, int epi, const gemm_device_params &dev)
{
    int d = 0;
    cudaGetDevice(&d);
    cudaDeviceProp prop;
    memset(&prop, 0, sizeof(prop));
    cudaGetDeviceProperties(&prop, d);
    char buf[512];
    snprintf(buf, sizeof(buf), "%lld|%lld|%lld|%d|%d|%s|%d|%s", (long long)M, (long long)N, (long long)K, dt, epi,
             prop.name, dev.sm_count, GEMM_LIB_VERSION);
    return buf;
}

int plan_tuned(int64_t M, int64_t N, int64_t K, int dt, int epi, gemm_plan_t *out, const TuneInputs *user)
{
    *out = nullptr;
    int rc = check_extents(M, N, K);
    if (rc) return rc;
    if (!valid_enums(dt, epi)) return set_error(GEMM_ERR_INVALID_ARG, "unknown dtype %d or epilogue %d", dt, epi);
    if ((rc = check_device_arch(nullptr))) return rc;
    gemm_device_params dev;
    if ((rc = query_params(&dev))) return rc;
    const char *dis = getenv("GEMM_DISABLE_AUTOTUNE");
    if (dis && dis[0] == '1') return make_plan(M, N, K, dt, epi, fixed_config(dt, dev), dev, nullptr, out);
    if (M == 0 || N == 0) return make_plan(M, N, K, dt, epi, fixed_config(dt, dev), dev, nullptr, out);
    const std::string key = cache_key(M, N, K, dt, epi, dev);
    gemm_config cfg;
    {
        std::lock_guard<std::mutex> lk(g_cache_mu);
        static std::string loaded_db;
        const char *dbp = db_path();
        if (dbp && loaded_db != dbp) {
            int64_t nl = 0;
            load_db_locked(dbp, &nl);   // a missing file is an empty database
            clear_error();
            loaded_db = dbp;
        }
        auto it = g_cache.find(key);
        if (it != g_cache.end()) {
            cfg = it->second;
            if (make_plan(M, N, K, dt, epi, cfg, dev, nullptr, out) == GEMM_OK) {
                ++g_hits;
                return GEMM_OK;
            }
            g_cache.erase(it);          // an entry the current limits reject is re-tuned
            clear_error();
        }
    }
    const char *mode = getenv("GEMM_TUNE_MODE");
    const bool exhaustive = mode && strcmp(mode, "exhaustive") == 0;
    const int topk = exhaustive ? 0 : std::max(1, env_int("GEMM_TUNE_TOPK", 24));
    std::vector<gemm_tune_row> rows;
    gemm_rank_stats stats;
    rc = tune(M, N, K, dt, epi, exhaustive ? GEMM_SEARCH_EXHAUSTIVE : GEMM_SEARCH_MODEL_TOPK, topk, 0, rows, stats,
              &cfg, nullptr, 0, user);
    if (rc) return rc;
    {
        std::lock_guard<std::mutex> lk(g_cache_mu);
        ++g_tunes;
        g_cache[key] = cfg;
        if (const char *dbp = db_path()) {
            if (FILE *f = fopen(dbp, "a")) {
                fputs(db_line(key, cfg).c_str(), f);
                fclose(f);
            }
        }
    }
    return make_plan(M, N, K, dt, epi, cfg, dev, nullptr, out);
}

// Plans by timing only the members of a given configuration list (no cache).
int plan_from_list(int64_t M, int64_t N, int64_t K, int dt, int epi, const gemm_config *list, int nlist,
                   gemm_plan_t *out)
{
    *out = nullptr;
    int rc = check_device_arch(nullptr);
    if (rc) return rc;
    gemm_device_params dev;
    if ((rc = query_params(&dev))) return rc;
    std::vector<gemm_tune_row> rows;
    gemm_rank_stats stats;
    gemm_config cfg;
    if (M == 0 || N == 0 || K == 0) {
        // Nothing to time: the first member that the rules accept.
        for (int i = 0; i < nlist; ++i)
            if (check_config(M, N, K, dt, epi, list[i], dev) == GEMM_FEASIBLE)
                return make_plan(M, N, K, dt, epi, list[i], dev, nullptr, out);
        return set_error(GEMM_ERR_UNSUPPORTED, "no configuration of the list runs this shape");
    }
    rc = tune(M, N, K, dt, epi, GEMM_SEARCH_EXHAUSTIVE, 0, 0, rows, stats, &cfg, list, nlist, nullptr);
    if (rc) return rc;
    return make_plan(M, N, K, dt, epi, cfg, dev, nullptr, out);
}

void cache_stats(int64_t *tunes, int64_t *hits, int64_t *entries);

// Ahead-of-time tuning of a list of shapes into the cache (and the file).
int tune_batch(const int64_t *mnk, int n, int dt, int epi, const char *path, int32_t *n_tuned)
{
    int64_t before = 0, after = 0;
    cache_stats(&before, nullptr, nullptr);
    for (int i = 0; i < n; ++i) {
        gemm_plan_t p = nullptr;
        const int rc = plan_tuned(mnk[3 * i], mnk[3 * i + 1], mnk[3 * i + 2], dt, epi, &p, nullptr);
        if (rc) return rc;
        destroy_plan(p);
    }
    cache_stats(&after, nullptr, nullptr);
    if (n_tuned) *n_tuned = (int32_t)(after - before);
    if (path) {
        int64_t written = 0;
        return cache_save(path, &written);
    }
    return GEMM_OK;
}

void cache_stats(int64_t *tunes, int64_t *hits, int64_t *entries)
{
    std::lock_guard<std::mutex> lk(g_cache_mu);
    if (tunes) *tunes = g_tunes;
    if (hits) *hits = g_hits;
    if (entries) *entries = (int64_t)g_cache.size();
}

void cache_clear()
{
    std::lock_guard<std::mutex> lk(g_cache_mu);
    g_cache.clear();
    g_tunes = 0;
    g_hits = 0;
}

int plan_explicit(int64_t M, int64_t N, int64_t K, int dt, int epi, const gemm_config &cfg, gemm_plan_t *out)
{
    *out = nullptr;
    int rc = check_device_arch(nullptr);
    if (rc) return rc;
    gemm_device_params dev;
    if ((rc = query_params(&dev))) return rc;
    return make_plan(M, N, K, dt, epi, cfg, dev, nullptr, out);
}

}  // namespace gemmgb
