// gemm_run_noalloc: the split-K bf16 GEMM with no allocation at all.
//
// Who needs it: callers that cannot call cudaMalloc.  Examples are code that
// runs inside a framework whose caching allocator owns the device memory (a
// raw cudaMalloc escapes its accounting and may synchronise the whole device),
// and services that reserve all device memory at start-up and must neither
// fail nor stall on an allocation while serving a request.  The planned path
// (gemm_plan / gemm_plan_with_config) allocates a status word, split-K arrival
// counters and the split-K partial-tile workspace with cudaMalloc; this entry
// point uses instead one fixed-size array compiled into the library.
//
// Scratch layout (g_noalloc_scratch):
//   [0, 256)                      status word (written when a device wait expires)
//   [256, 256 + 4·MAX_TILES)      split-K arrival counters, one per output tile
//   [NOALLOC_CTL_BYTES, + WS)     split-K partial tiles (fp32)
// Every GPU that loads the library holds the whole array until the process exits.
// All calls share it and it keeps the previous call's contents; each call clears
// the status word and the counters it uses on its stream before the kernel runs,
// and calls whose work overlaps on the GPU (different streams, or several host
// threads) race on the array.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "gemm_internal.h"

// The scratch itself: file scope, fixed size, zero at module load.
static __device__ __align__(256) unsigned char g_noalloc_scratch[256 + (size_t)GEMM_NOALLOC_MAX_TILES * 4 +
                                                                  (size_t)GEMM_NOALLOC_WORKSPACE_BYTES];

namespace gemmgb {

int query_params(gemm_device_params *d);      // runtime.cpp
extern std::atomic<int64_t> g_timeout_ns;     // runtime.cpp
extern std::atomic<int32_t> g_debug_stall;    // runtime.cpp
extern std::atomic<int32_t> g_check;          // runtime.cpp

namespace {

constexpr size_t kNoallocCtlBytes = 256 + (size_t)GEMM_NOALLOC_MAX_TILES * 4;
static_assert(kNoallocCtlBytes % 256 == 0, "workspace must start 256-byte aligned");
static_assert(sizeof(g_noalloc_scratch) == kNoallocCtlBytes + (size_t)GEMM_NOALLOC_WORKSPACE_BYTES, "layout");

constexpr int kMaxDevices = 64;

struct DeviceSetup {
    bool ready = false;
    unsigned char *scratch = nullptr;   // device address of g_noalloc_scratch
    gemm_device_params params{};
};

std::mutex g_setup_mu;
DeviceSetup g_setup[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode_fn = nullptr;

// Set-up of the current device, done once: the array's device address (the
// host-side symbol is only a stand-in and must not be given to a kernel), the
// device parameters, the kernel's shared-memory limit and the driver's tensor-
// map encoder.  None of it allocates memory.
int setup_current_device(const DeviceSetup **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return set_error(GEMM_ERR_NO_DEVICE, "no CUDA device: %s", cudaGetErrorString(e));
    }
    if (dev < 0 || dev >= kMaxDevices)
        return set_error(GEMM_ERR_UNSUPPORTED, "device index %d is beyond the %d supported", dev, kMaxDevices);
    std::lock_guard<std::mutex> lk(g_setup_mu);
    DeviceSetup &s = g_setup[dev];
    if (!s.ready) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (major != 10 || minor != 3)
            return set_error(GEMM_ERR_UNSUPPORTED, "kernels are built for sm_103a; device %d is sm_%d%d", dev, major,
                             minor);
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || ptr == nullptr)
            return set_error(GEMM_ERR_CUDA, "cudaGetSymbolAddress(no-allocation scratch): %s", cudaGetErrorString(e));
        int rc = query_params(&s.params);
        if (rc) return rc;
        e = set_kernel_smem_limit(GEMM_BF16, (int)s.params.smem_per_block);
        if (e != cudaSuccess)
            return set_error(GEMM_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        if (!g_encode_fn) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr)
                return set_error(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
            g_encode_fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        s.scratch = static_cast<unsigned char *>(ptr);
        s.ready = true;
    }
    *out = &s;
    return GEMM_OK;
}

// Row-major bf16 [outer, inner] matrix described for TMA, box [box_outer, box_inner].
int encode_bf16(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
                uint32_t box_outer, CUtensorMapSwizzle sw, CUtensorMapL2promotion l2)
{
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode_fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
                             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(GEMM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return GEMM_OK;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace
}  // namespace gemmgb

using namespace gemmgb;

extern "C" int gemm_run_noalloc(int64_t M, int64_t N, int64_t K, gemm_epilogue epi, const gemm_config *cfg,
                                const void *A, const void *B, const void *bias, void *C, gemm_stream_t stream)
{
    clear_error();
    const int64_t lim = (int64_t)1 << 31;
    if (!cfg || M < 0 || N < 0 || K < 0 || M >= lim || N >= lim || K >= lim || epi < GEMM_EPI_NONE ||
        epi > GEMM_EPI_BIAS_GELU)
        return set_error(GEMM_ERR_INVALID_ARG, "gemm_run_noalloc: bad extents, epilogue or null config");
    const DeviceSetup *ds = nullptr;
    int rc = setup_current_device(&ds);
    if (rc) return rc;
    const gemm_config c = *cfg;
    const int reason = check_config(M, N, K, GEMM_BF16, epi, c, ds->params);
    if (reason == GEMM_REASON_ALIGN)
        return set_error(GEMM_ERR_MISALIGNED, "K=%lld / N=%lld: %s", (long long)K, (long long)N, reason_text(reason));
    if (reason != GEMM_FEASIBLE) return set_error(GEMM_ERR_INFEASIBLE, "config rejected: %s", reason_text(reason));
    if (c.cta_group != 1)
        return set_error(GEMM_ERR_UNSUPPORTED, "gemm_run_noalloc runs single-CTA tiles only (cta_group 1)");
    if (M == 0 || N == 0) return GEMM_OK;
    const int64_t rows = c.swap_ab ? N : M, cols = c.swap_ab ? M : N;
    const int64_t tiles_m = cdiv(rows, c.bm), tiles_n = cdiv(cols, c.bn), tiles = tiles_m * tiles_n;
    const uint64_t ws_bytes = c.split_k > 1 ? (uint64_t)tiles * c.split_k * c.bm * c.bn * 4u : 0u;
    if (tiles > GEMM_NOALLOC_MAX_TILES || ws_bytes > (uint64_t)GEMM_NOALLOC_WORKSPACE_BYTES)
        return set_error(GEMM_ERR_INVALID_ARG,
                         "gemm_run_noalloc: %lld tiles and %llu workspace bytes exceed the fixed scratch "
                         "(%d tiles, %u bytes); use fewer tiles or a smaller split_k, or gemm_plan",
                         (long long)tiles, (unsigned long long)ws_bytes, GEMM_NOALLOC_MAX_TILES,
                         (unsigned)GEMM_NOALLOC_WORKSPACE_BYTES);
    if (!C || (K > 0 && (!A || !B))) return set_error(GEMM_ERR_INVALID_ARG, "null A, B or C");
    if (epi != GEMM_EPI_NONE && !bias) return set_error(GEMM_ERR_INVALID_ARG, "bias is required by the epilogue");
    if ((K > 0 && (!aligned16(A) || !aligned16(B))) || !aligned16(C) || (epi != GEMM_EPI_NONE && !aligned16(bias)))
        return set_error(GEMM_ERR_MISALIGNED, "A, B, C and bias must be 16-byte aligned");

    // Tensor maps: A [M, K] K-major; B [K, N] read MN-major in place; C stores.
    const int span = span_elems(GEMM_BF16);
    CUtensorMap ma, mb, mc;
    memset(&ma, 0, sizeof(ma));
    memset(&mb, 0, sizeof(mb));
    if (K > 0) {
        CUtensorMap *am = c.swap_ab ? &mb : &ma;
        CUtensorMap *bmap = c.swap_ab ? &ma : &mb;
        rc = encode_bf16(am, A, K, M, span, c.swap_ab ? c.bn : c.bm, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
        if (!rc)
            rc = encode_bf16(bmap, B, N, K, span, c.bk, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
        if (rc) return rc;
    }
    if (!c.swap_ab)
        rc = encode_bf16(&mc, C, N, M, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE);
    else
        rc = encode_bf16(&mc, C, N, M, 32, 16, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE);
    if (rc) return rc;

    const Layout L = layout_of(c, GEMM_BF16);
    // The same launch record as a plan of this configuration (B read MN-major
    // in place); the split-K exchange goes through the last-arriver route,
    // whose counters this call clears below.
    KernelParams k = kernel_params_of(M, N, K, GEMM_BF16, epi, c, false);
    k.bias = epi != GEMM_EPI_NONE ? bias : nullptr;
    k.status = reinterpret_cast<int32_t *>(ds->scratch);
    k.counters = reinterpret_cast<int32_t *>(ds->scratch + 256);
    k.workspace = reinterpret_cast<float *>(ds->scratch + kNoallocCtlBytes);
    k.timeout_ns = g_timeout_ns.load();
    k.debug_stall = g_debug_stall.load();

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // The status word and this call's counters must start at zero.
    cudaError_t e = cudaMemsetAsync(ds->scratch, 0, 256 + (size_t)tiles * 4, s);
    if (e != cudaSuccess) return set_error(GEMM_ERR_CUDA, "clearing the scratch counters: %s", cudaGetErrorString(e));
    const int grid = (int)std::min<int64_t>(k.num_units, ds->params.sm_count);
    const int64_t one_per_sm = ds->params.smem_per_block / 2 + 1024;
    const int smem = (int)std::min<int64_t>(ds->params.smem_per_block, std::max<int64_t>(L.smem_total, one_per_sm));
    e = launch_gemm(GEMM_BF16, ma, mb, mc, nullptr, nullptr, k, grid, smem, s);
    if (e != cudaSuccess) return set_error(GEMM_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
    if (g_check.load()) {
        // Checked runs (GEMM_CHECK / gemm_debug_set(4, 1)): wait for the kernel
        // and read the status word straight from the array, without allocating.
        e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return set_error(GEMM_ERR_CUDA, "cudaStreamSynchronize (checked run): %s",
                                               cudaGetErrorString(e));
        int32_t st = 0;
        e = cudaMemcpyFromSymbol(&st, g_noalloc_scratch, sizeof(st), 0, cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return set_error(GEMM_ERR_CUDA, "reading the status word: %s", cudaGetErrorString(e));
        if (st != 0)
            return set_error(GEMM_ERR_TIMEOUT, "a device wait expired (site %d); the kernel returned early", st);
    }
    return GEMM_OK;
}
