// Internal declarations shared by the host-side translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "../../include/gemm_gb300.h"
#include "kernel_params.h"

#define GEMM_LIB_VERSION "gb300-tcgen05-gemm 0.1.0"

namespace gemmgb {

constexpr int kThreadsPerCta = 320;
constexpr int kTmemColumns = 512;
constexpr int kAuxSmem = 2048;     // barriers and flags (1 KB) + 1 KB of base-alignment slack
constexpr int kMaxStages = 16;
constexpr int kMaxSplitK = 16;

// Gated epilogues: C [M, N/2] = act(gate) ⊙ up over a fused [K, N] weight.
inline bool is_glu(int epi) { return epi >= GEMM_EPI_BIAS_REGLU && epi <= GEMM_EPI_BIAS_SWIGLU; }
inline bool is_residual(int epi) { return epi >= GEMM_EPI_BIAS_RESIDUAL && epi <= GEMM_EPI_BIAS_GELU_RESIDUAL; }

// FP8 operands, plain (one tensor scale) or block-scaled (MX).
inline bool is_fp8(int dt) { return dt == GEMM_FP8_E4M3 || dt == GEMM_MXFP8_E4M3; }
// Operand element size, and the size of C, bias and R (FP8 operands give bf16).
inline int elt_bytes(int dt) { return dt == GEMM_BF16 ? 2 : is_fp8(dt) ? 1 : 4; }
inline int out_elt_bytes(int dt) { return dt == GEMM_FP32_TF32 ? 4 : 2; }
inline int span_elems(int dt) { return 128 / elt_bytes(dt); }
// Whether B is read MN-major in place: bf16 always; FP8 when B's rows (N
// bytes) meet TMA's 16-byte stride rule, else from a K-major copy, as fp32.
inline bool b_in_place(int dt, int64_t N) { return dt == GEMM_BF16 || (is_fp8(dt) && N % 16 == 0); }
// MX scales: one atom holds 128 rows x 128 K (four 32-element blocks a row) in
// 512 bytes; the packed arrays pad rows and K to multiples of 256 (two atoms).
constexpr int kMxAtomBytes = 512;
inline int64_t mx_row_atoms(int64_t rows) { return 2 * ((rows + 255) / 256); }
inline int64_t mx_k_atoms(int64_t K) { return 2 * ((K + 255) / 256); }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Shared-memory and TMEM layout of one configuration.
struct Layout {
    uint32_t a_stage_bytes, b_stage_bytes, stage_bytes;
    uint32_t staging_buf_bytes, staging_total;
    uint32_t off_b, off_staging, off_bar;
    uint32_t smem_total;              // bytes the kernel needs, slack included
    uint32_t acc_cols, n_acc, tmem_cols;
    // MX scales: bytes a stage stages (A's atoms, then B's) at off_sf, and the
    // TMEM columns a stage's scales occupy, one slot per stage from sc_col0.
    uint32_t sf_stage_bytes, off_sf, sc_stage_cols, sc_col0;
};
Layout layout_of(const gemm_config &c, int dt);
int max_stages_for(int bm, int bn, int bk, int dt, int swap_ab, int64_t smem_per_block, int cta_group);
bool cluster_reduce_fits(const gemm_config &c, int dt);
// Bytes of partials the busiest owner of a cluster split-K receives (16 KB slots).
uint32_t cluster_recv_bytes(const gemm_config &c);

// Launch record of configuration c for C = act(A·B + bias) on (M, N, K) in
// dtype dt, with `act` the kernel's bias/activation code (0 none, 1 bias, 2
// ReLU, 3 GELU) and B read from a K-major copy when `b_kmajor`: extents,
// schedule, operand majorness, the tcgen05 instruction descriptor and the
// shared-memory / TMEM layout, with alpha = 1.  Pointers, the split-K route
// and the run's debug fields are left zero for the caller.
KernelParams kernel_params_of(int64_t M, int64_t N, int64_t K, int dt, int act, const gemm_config &c,
                              bool b_kmajor);

// Operands a caller lends the tuner (device pointers in the layouts gemm_run and
// gemm_run_mx take; SA and SB packed MX scales, block-scaled plans only): the
// candidates are timed on copies of them instead of on synthetic fills.
struct TuneInputs {
    const void *A, *B, *bias, *SA, *SB;
};

// Host logic (planner.cpp)
void params_default(gemm_device_params *d);
void params_workshop(gemm_device_params *d);
int check_config(int64_t M, int64_t N, int64_t K, int dt, int epi, const gemm_config &c,
                 const gemm_device_params &d);
std::vector<gemm_config> enumerate(int64_t M, int64_t N, int64_t K, int dt, int epi,
                                   const gemm_device_params &d);
gemm_config fixed_config(int dt, const gemm_device_params &d);
gemm_model_terms predict(int64_t M, int64_t N, int64_t K, int dt, int epi, const gemm_config &c,
                         const gemm_device_params &d);
gemm_rank_stats rank_agreement(const double *pred, const double *meas, int n);
int select_config_set(const double *t, int ns, int nc, int max_set, int32_t *chosen, int32_t *n_chosen,
                      double *mean_slowdown, double *worst_slowdown);
const char *reason_text(int reason);

// Errors (capi.cpp)
int set_error(int code, const char *fmt, ...);
void clear_error();

// Kernel launch (gemm_kernel.cu)
cudaError_t kernel_attributes(int dt, int *num_regs, int *max_threads);
cudaError_t set_kernel_smem_limit(int dt, int bytes);
cudaError_t max_active_clusters(int dt, int a_mn, int b_mn, int cg, int cluster, int smem_bytes, int *out);
cudaError_t launch_gemm(int dt, const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &c,
                        const CUtensorMap *sa, const CUtensorMap *sb, const KernelParams &p, int grid, int smem_bytes,
                        cudaStream_t stream);
cudaError_t launch_transpose(const void *src, void *dst, int64_t rows, int64_t cols, int elt, cudaStream_t stream);
cudaError_t launch_fill_random(void *dst, int64_t n, int dt, float scale, uint32_t seed, int dist,
                               cudaStream_t stream);
cudaError_t launch_mx_pack(const uint8_t *src, int64_t rows, int64_t K, int b_side, uint8_t *dst,
                           cudaStream_t stream);

}  // namespace gemmgb
