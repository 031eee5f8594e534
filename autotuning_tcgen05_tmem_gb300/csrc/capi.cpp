// extern "C" boundary of the library (declared in include/gemm_gb300.h).
// Argument checking and marshalling only; the work is in planner.cpp,
// runtime.cpp and gemm_kernel.cu.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <string>
#include <vector>

#include "gemm_internal.h"
#include "schedule.h"

namespace gemmgb {

static thread_local std::string t_last_error;

int set_error(int code, const char *fmt, ...)
{
    char buf[1024];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return code;
}

void clear_error() { t_last_error.clear(); }

// runtime.cpp
extern std::atomic<int64_t> g_timeout_ns;
extern std::atomic<int32_t> g_debug_stall;
extern std::atomic<int32_t> g_b_route;
extern std::atomic<int32_t> g_split_route;
extern std::atomic<int32_t> g_check;
extern std::atomic<int64_t> g_share_poll;
extern std::atomic<int32_t> g_tune_fill;
extern std::atomic<int32_t> g_span3d;
int query_params(gemm_device_params *d);
int model_params_load(const char *path, gemm_device_params *out);
int plan_tuned(int64_t M, int64_t N, int64_t K, int dt, int epi, gemm_plan_t *out, const TuneInputs *user);
int plan_explicit(int64_t M, int64_t N, int64_t K, int dt, int epi, const gemm_config &cfg, gemm_plan_t *out);
int run_plan(gemm_plan_t p, const void *A, const void *B, const void *bias, void *C, cudaStream_t stream);
int run_plan_ex(gemm_plan_t p, const void *A, const void *B, const void *bias, const void *R, void *C,
                cudaStream_t stream);
int run_plan_mx(gemm_plan_t p, const void *A, const void *SA, const void *B, const void *SB, const void *bias,
                const void *R, void *C, cudaStream_t stream);
int mx_pack_scales(const void *scales, int64_t rows, int64_t K, int b_side, void *packed, cudaStream_t stream);
int run_host(gemm_plan_t p, const void *A, const void *B, const void *bias, void *C, cudaStream_t stream);
int run_host_many(gemm_plan_t p, int n, const void *const *A, const void *const *B, const void *const *bias,
                  void *const *C, cudaStream_t stream);
int plan_status(gemm_plan_t p);
int plan_config(gemm_plan_t p, gemm_config *out);
int plan_launch_info(gemm_plan_t p, gemm_launch_info *out);
int plan_set_scale(gemm_plan_t p, float alpha);
int plan_set_independent_operands(gemm_plan_t p, int32_t mask);
void destroy_plan(gemm_plan_t p);
int tune(int64_t M, int64_t N, int64_t K, int dt, int epi, int mode, int topk, uint64_t seed,
         std::vector<gemm_tune_row> &rows, gemm_rank_stats &stats, gemm_config *winner,
         const gemm_config *list, int nlist, const TuneInputs *user);
int plan_from_list(int64_t M, int64_t N, int64_t K, int dt, int epi, const gemm_config *list, int nlist,
                   gemm_plan_t *out);
int tune_batch(const int64_t *mnk, int n, int dt, int epi, const char *path, int32_t *n_tuned);
void cache_stats(int64_t *tunes, int64_t *hits, int64_t *entries);
void cache_clear();
int cache_save(const char *path, int64_t *n);
int cache_load(const char *path, int64_t *n);

}  // namespace gemmgb

using namespace gemmgb;

struct gemm_plan_s;  // defined in runtime.cpp
extern "C" {

const char *gemm_version(void) { return GEMM_LIB_VERSION; }

const char *gemm_last_error(void) { return t_last_error.c_str(); }

void gemm_device_params_default(gemm_device_params *out)
{
    if (out) params_default(out);
}

void gemm_device_params_workshop(gemm_device_params *out)
{
    if (out) params_workshop(out);
}

static bool enums_ok(int dt, int epi)
{
    return dt >= GEMM_BF16 && dt <= GEMM_MXFP8_E4M3 && epi >= GEMM_EPI_NONE && epi <= GEMM_EPI_BIAS_SWIGLU;
}

int gemm_check_config(int64_t M, int64_t N, int64_t K, gemm_dtype dtype, gemm_epilogue epi, const gemm_config *cfg,
                      const gemm_device_params *dev)
{
    clear_error();
    if (!cfg || !dev || !enums_ok(dtype, epi) || M < 0 || N < 0 || K < 0)
        return set_error(GEMM_ERR_INVALID_ARG, "gemm_check_config: bad argument");
    return check_config(M, N, K, dtype, epi, *cfg, *dev);
}

int gemm_enumerate(int64_t M, int64_t N, int64_t K, gemm_dtype dtype, gemm_epilogue epi,
                   const gemm_device_params *dev, gemm_config *out, int32_t cap, int32_t *n)
{
    clear_error();
    if (!dev || !n || !enums_ok(dtype, epi) || M < 0 || N < 0 || K < 0 || cap < 0 || (cap > 0 && !out))
        return set_error(GEMM_ERR_INVALID_ARG, "gemm_enumerate: bad argument");
    const std::vector<gemm_config> v = enumerate(M, N, K, dtype, epi, *dev);
    *n = (int32_t)v.size();
    for (int32_t i = 0; i < cap && i < (int32_t)v.size(); ++i) out[i] = v[i];
    return GEMM_OK;
}

int gemm_fixed_config(gemm_dtype dtype, const gemm_device_params *dev, gemm_config *out)
{
    clear_error();
    if (!dev || !out || !enums_ok(dtype, 0)) return set_error(GEMM_ERR_INVALID_ARG, "gemm_fixed_config: bad argument");
    *out = fixed_config(dtype, *dev);
    return GEMM_OK;
}

int gemm_model_predict(int64_t M, int64_t N, int64_t K, gemm_dtype dtype, gemm_epilogue epi, const gemm_config *cfg,
                       const gemm_device_params *dev, gemm_model_terms *out)
{
    clear_error();
    if (!cfg || !dev || !out || !enums_ok(dtype, epi) || M < 0 || N < 0 || K < 0 || cfg->bm <= 0 || cfg->bn <= 0 ||
        cfg->bk <= 0 || cfg->stages <= 0 || cfg->split_k <= 0 || cfg->group <= 0 || dev->sm_count <= 0)
        return set_error(GEMM_ERR_INVALID_ARG, "gemm_model_predict: bad argument");
    *out = predict(M, N, K, dtype, epi, *cfg, *dev);
    return GEMM_OK;
}

int gemm_rank_agreement(const double *predicted, const double *measured, int32_t n, gemm_rank_stats *out)
{
    clear_error();
    if (!predicted || !measured || !out || n < 2) return set_error(GEMM_ERR_INVALID_ARG, "gemm_rank_agreement: bad argument");
    *out = rank_agreement(predicted, measured, n);
    return GEMM_OK;
}

int gemm_schedule_unit(int64_t unit, int32_t tiles_m, int32_t tiles_n, int32_t split_k, int32_t raster, int32_t group,
                       int32_t num_kb, int32_t *tile_m, int32_t *tile_n, int32_t *split, int32_t *kb_begin,
                       int32_t *kb_end)
{
    clear_error();
    if (tiles_m <= 0 || tiles_n <= 0 || split_k <= 0 || group <= 0 || num_kb < 0 || (raster != 0 && raster != 1) ||
        unit < 0 || unit >= (int64_t)tiles_m * tiles_n * split_k)
        return set_error(GEMM_ERR_INVALID_ARG, "gemm_schedule_unit: bad argument");
    const SchedUnit u = schedule_unit(unit, tiles_m, tiles_n, split_k, raster, group, num_kb);
    if (tile_m) *tile_m = u.tile_m;
    if (tile_n) *tile_n = u.tile_n;
    if (split) *split = u.split;
    if (kb_begin) *kb_begin = u.kb_begin;
    if (kb_end) *kb_end = u.kb_end;
    return GEMM_OK;
}

int gemm_device_params_query(gemm_device_params *out)
{
    clear_error();
    if (!out) return set_error(GEMM_ERR_INVALID_ARG, "null output");
    return query_params(out);
}

int gemm_plan(int64_t M, int64_t N, int64_t K, gemm_dtype dtype, gemm_epilogue epi, gemm_plan_t *out)
{
    clear_error();
    if (!out) return set_error(GEMM_ERR_INVALID_ARG, "null output");
    return plan_tuned(M, N, K, dtype, epi, out, nullptr);
}

int gemm_plan_tuned_on(int64_t M, int64_t N, int64_t K, gemm_dtype dtype, gemm_epilogue epi, const void *A,
                       const void *SA, const void *B, const void *SB, const void *bias, gemm_plan_t *out)
{
    clear_error();
    if (!out) return set_error(GEMM_ERR_INVALID_ARG, "null output");
    const TuneInputs in{A, B, bias, SA, SB};
    return plan_tuned(M, N, K, dtype, epi, out, &in);
}

int gemm_plan_with_config(int64_t M, int64_t N, int64_t K, gemm_dtype dtype, gemm_epilogue epi,
                          const gemm_config *cfg, gemm_plan_t *out)
{
    clear_error();
    if (!out || !cfg) return set_error(GEMM_ERR_INVALID_ARG, "null argument");
    return plan_explicit(M, N, K, dtype, epi, *cfg, out);
}

int gemm_plan_config(gemm_plan_t plan, gemm_config *out)
{
    clear_error();
    return plan_config(plan, out);
}

int gemm_plan_set_scale(gemm_plan_t plan, float alpha)
{
    clear_error();
    return plan_set_scale(plan, alpha);
}

int gemm_plan_launch_info(gemm_plan_t plan, gemm_launch_info *out)
{
    clear_error();
    if (!plan || !out) return set_error(GEMM_ERR_INVALID_ARG, "null argument");
    return plan_launch_info(plan, out);
}

int gemm_run(gemm_plan_t plan, const void *A, const void *B, const void *bias, void *C, gemm_stream_t stream)
{
    return run_plan(plan, A, B, bias, C, reinterpret_cast<cudaStream_t>(stream));
}

int gemm_run_ex(gemm_plan_t plan, const void *A, const void *B, const void *bias, const void *R, void *C,
                gemm_stream_t stream)
{
    return run_plan_ex(plan, A, B, bias, R, C, reinterpret_cast<cudaStream_t>(stream));
}

int gemm_plan_set_independent_operands(gemm_plan_t plan, int32_t mask)
{
    clear_error();
    return plan_set_independent_operands(plan, mask);
}

int gemm_model_params_load(const char *path, gemm_device_params *dev)
{
    clear_error();
    return model_params_load(path, dev);
}

int gemm_run_mx(gemm_plan_t plan, const void *A, const void *SA, const void *B, const void *SB, const void *bias,
                const void *R, void *C, gemm_stream_t stream)
{
    return run_plan_mx(plan, A, SA, B, SB, bias, R, C, reinterpret_cast<cudaStream_t>(stream));
}

int64_t gemm_mx_scales_bytes(int64_t rows, int64_t K)
{
    if (rows < 0 || K < 0) return 0;
    return mx_row_atoms(rows) * mx_k_atoms(K) * kMxAtomBytes;
}

int gemm_mx_pack_scales(const void *scales, int64_t rows, int64_t K, int32_t b_side, void *packed,
                        gemm_stream_t stream)
{
    clear_error();
    return mx_pack_scales(scales, rows, K, b_side, packed, reinterpret_cast<cudaStream_t>(stream));
}

int gemm_run_host(gemm_plan_t plan, const void *A, const void *B, const void *bias, void *C, gemm_stream_t stream)
{
    clear_error();
    return run_host(plan, A, B, bias, C, reinterpret_cast<cudaStream_t>(stream));
}

int gemm_run_host_many(gemm_plan_t plan, int32_t n, const void *const *A, const void *const *B,
                       const void *const *bias, void *const *C, gemm_stream_t stream)
{
    clear_error();
    return run_host_many(plan, n, A, B, bias, C, reinterpret_cast<cudaStream_t>(stream));
}

int gemm_plan_status(gemm_plan_t plan)
{
    clear_error();
    return plan_status(plan);
}

void gemm_plan_destroy(gemm_plan_t plan) { destroy_plan(plan); }

static int tune_into(int64_t M, int64_t N, int64_t K, int dtype, int epi, int mode, int32_t k, uint64_t seed,
                     gemm_tune_row *rows, int32_t cap, int32_t *n_rows, gemm_rank_stats *stats,
                     const TuneInputs *user = nullptr)
{
    if (!n_rows || cap < 0 || (cap > 0 && !rows)) return set_error(GEMM_ERR_INVALID_ARG, "gemm_tune: bad argument");
    std::vector<gemm_tune_row> v;
    gemm_rank_stats s;
    const int rc = tune(M, N, K, dtype, epi, mode, k, seed, v, s, nullptr, nullptr, 0, user);
    if (rc) return rc;
    int32_t i = 0;
    for (; i < cap && i < (int32_t)v.size(); ++i) rows[i] = v[i];
    *n_rows = i;
    if (stats) *stats = s;
    return GEMM_OK;
}

int gemm_tune(int64_t M, int64_t N, int64_t K, gemm_dtype dtype, gemm_epilogue epi, int32_t topk, gemm_tune_row *rows,
              int32_t cap, int32_t *n_rows, gemm_rank_stats *stats)
{
    clear_error();
    return tune_into(M, N, K, dtype, epi, topk > 0 ? GEMM_SEARCH_MODEL_TOPK : GEMM_SEARCH_EXHAUSTIVE, topk, 0, rows,
                     cap, n_rows, stats);
}

int gemm_tune_on(int64_t M, int64_t N, int64_t K, gemm_dtype dtype, gemm_epilogue epi, const void *A, const void *SA,
                 const void *B, const void *SB, const void *bias, int32_t topk, gemm_tune_row *rows, int32_t cap,
                 int32_t *n_rows, gemm_rank_stats *stats)
{
    clear_error();
    const TuneInputs in{A, B, bias, SA, SB};
    return tune_into(M, N, K, dtype, epi, topk > 0 ? GEMM_SEARCH_MODEL_TOPK : GEMM_SEARCH_EXHAUSTIVE, topk, 0, rows,
                     cap, n_rows, stats, &in);
}

int gemm_tune_search(int64_t M, int64_t N, int64_t K, gemm_dtype dtype, gemm_epilogue epi, gemm_search mode,
                     int32_t k, uint64_t seed, gemm_tune_row *rows, int32_t cap, int32_t *n_rows,
                     gemm_rank_stats *stats)
{
    clear_error();
    if (mode < GEMM_SEARCH_EXHAUSTIVE || mode > GEMM_SEARCH_RANDOM_K || (mode != GEMM_SEARCH_EXHAUSTIVE && k < 1))
        return set_error(GEMM_ERR_INVALID_ARG, "gemm_tune_search: bad mode or budget");
    return tune_into(M, N, K, dtype, epi, mode, k, seed, rows, cap, n_rows, stats);
}

int gemm_cache_save(const char *path, int64_t *n_written)
{
    clear_error();
    return cache_save(path, n_written);
}

int gemm_cache_load(const char *path, int64_t *n_loaded)
{
    clear_error();
    return cache_load(path, n_loaded);
}

int gemm_cache_stats(int64_t *tunes, int64_t *hits, int64_t *entries)
{
    cache_stats(tunes, hits, entries);
    return GEMM_OK;
}

void gemm_cache_clear(void) { cache_clear(); }

int gemm_select_config_set(const double *times, int32_t n_shapes, int32_t n_configs, int32_t max_set,
                           int32_t *chosen, int32_t *n_chosen, double *mean_slowdown, double *worst_slowdown)
{
    clear_error();
    if (n_shapes < 0 || n_configs < 0 || max_set < 0 || !n_chosen || (max_set > 0 && !chosen) ||
        ((int64_t)n_shapes * n_configs > 0 && !times))
        return set_error(GEMM_ERR_INVALID_ARG, "gemm_select_config_set: bad argument");
    return select_config_set(times, n_shapes, n_configs, std::min(max_set, n_configs), chosen, n_chosen,
                             mean_slowdown, worst_slowdown);
}

int gemm_plan_from_list(int64_t M, int64_t N, int64_t K, gemm_dtype dtype, gemm_epilogue epi,
                        const gemm_config *list, int32_t n, gemm_plan_t *out)
{
    clear_error();
    if (!out || n < 0 || (n > 0 && !list)) return set_error(GEMM_ERR_INVALID_ARG, "gemm_plan_from_list: bad argument");
    return plan_from_list(M, N, K, dtype, epi, list, n, out);
}

int gemm_tune_batch(const int64_t *mnk, int32_t n, gemm_dtype dtype, gemm_epilogue epi, const char *db_path,
                    int32_t *n_tuned)
{
    clear_error();
    if (n < 0 || (n > 0 && !mnk)) return set_error(GEMM_ERR_INVALID_ARG, "gemm_tune_batch: bad argument");
    return tune_batch(mnk, n, dtype, epi, db_path, n_tuned);
}

int gemm_debug_set(int32_t what, int64_t value)
{
    clear_error();
    if (what == 0) {
        if (value <= 0) return set_error(GEMM_ERR_INVALID_ARG, "wait limit must be positive");
        g_timeout_ns.store(value);
        return GEMM_OK;
    }
    if (what == 1) {
        g_debug_stall.store(value ? 1 : 0);
        return GEMM_OK;
    }
    if (what == 2) {
        if (value < 0 || value > 2) return set_error(GEMM_ERR_INVALID_ARG, "B route must be 0, 1 or 2");
        g_b_route.store((int32_t)value);
        return GEMM_OK;
    }
    if (what == 3) {
        if (value < 0 || value > 1) return set_error(GEMM_ERR_INVALID_ARG, "split-K route must be 0 or 1");
        g_split_route.store((int32_t)value);
        return GEMM_OK;
    }
    if (what == 4) {
        g_check.store(value ? 1 : 0);
        return GEMM_OK;
    }
    if (what == 5) {
        if (value < 0) return set_error(GEMM_ERR_INVALID_ARG, "the share wait must be >= 0 cycles");
        g_share_poll.store(value);
        return GEMM_OK;
    }
    if (what == 6) {
        if (value < 0 || value > 1) return set_error(GEMM_ERR_INVALID_ARG, "tuning fill must be 0 or 1");
        g_tune_fill.store((int32_t)value);
        return GEMM_OK;
    }
    if (what == 7) {
        if (value < 0 || value > 1) return set_error(GEMM_ERR_INVALID_ARG, "span copies must be 0 or 1");
        g_span3d.store((int32_t)value);
        return GEMM_OK;
    }
    return set_error(GEMM_ERR_INVALID_ARG, "unknown debug control %d", what);
}

}  // extern "C"
