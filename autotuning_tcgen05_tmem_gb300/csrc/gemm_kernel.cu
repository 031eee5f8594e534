// Persistent, warp-specialised tcgen05 GEMM for sm_103a:
//   C = act(alpha·(A·B) + bias) (+ R),  operands bf16, fp32 (read as tf32),
//   FP8 E4M3, or block-scaled FP8 (MX: E4M3 with an E8M0 scale per 32 elements
//   of K); with FP8 operands C, bias and R are bf16.
//
// What the pages fix and how this kernel realises it on GB300:
//   * "Tile Selection: Cost Models Against Measurement", "The structure of the
//     search space": one output tile [BM, BN] per work unit; the reduction runs
//     in steps of BK, each step staging a [BM, BK] panel of A and a [BK, BN]
//     panel of B in shared memory.  Here the per-thread tile of the page is
//     replaced by a tensor-memory (TMEM) accumulator written by tcgen05.mma.
//   * "Tiling the hierarchy", double buffering: loads overlap compute only when
//     they are asynchronous; a deeper ring absorbs latency.  Here TMA
//     (cp.async.bulk.tensor) fills an S-stage ring guarded by mbarriers, and the
//     accumulator itself is double-buffered in TMEM so the epilogue of one tile
//     overlaps the main loop of the next.
//   * "Tiling the hierarchy", fusion: the elementwise epilogue (bias, ReLU,
//     GELU) is fused onto the GEMM: TMEM -> registers -> shared staging -> TMA
//     store, so C is written once, coalesced.
//   * "Compilers and Kernel Languages": pipeline depth, split-K and tile order
//     are runtime choices of this kernel (stages, split_k, raster/group).
//
// Roles (320 threads): warp 0 issues TMA loads and warp 1 owns TMEM and issues
// tcgen05.mma (one elected lane each, the warp walking the schedule converged);
// warps 2..9 (256 threads) drain the accumulator, each reading the 32 TMEM
// lanes of its sub-partition (warp % 4), two warps per sub-partition.  With
// CG = 2 two consecutive CTAs share a 256-row tile (cta_group::2): each holds
// 128 rows and half of B, and the first CTA's MMA warp issues for both.
//
// Split-K: the K slices of a tile either exchange fp32 partial tiles through
// global memory (a cooperative fix-up when all slices are resident, each slice
// finalising its share; else the last slice to arrive finalises the tile), or,
// when the slices of a tile form one thread-block cluster, push them into the
// owning CTA's shared memory with st.async (distributed shared memory).  Every
// route adds the partials in slice order, so all give the same bits.
//
// Every mbarrier wait is bounded: after the limit the waiting role writes a
// code to the status word, raises a CTA-wide abort flag and returns; the other
// roles see the flag, the CTA waits (bounded) for its own copies and MMAs in
// flight, frees TMEM and exits.  Nothing traps.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "kernel_params.h"
#include "schedule.h"

namespace gemmgb {
namespace {

constexpr int kEpiWarps = 8;                    // two per TMEM sub-partition
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = 64 + kEpiThreads;      // producer warp + MMA warp + epilogue

// ---------------------------------------------------------------------------
// Inline-PTX primitives
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Non-blocking probe with cluster-scope acquire, for barriers that CTAs of
// the cluster arrive on remotely or that st.async from them completes (a
// suspended try_wait is not reliably woken by those remote arrivals).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Address of the same shared-memory location in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_u32(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Arrivals on another CTA's barrier (default release.cta semantics: what they
// order is either async-proxy traffic that completes on the barrier itself or
// tcgen05 work fenced before the arrival).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx_remote(uint32_t cluster_addr, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cluster.b64 _, [%0], %1;" ::"r"(cluster_addr), "r"(bytes)
                 : "memory");
}

// 16-byte store into another CTA's shared memory; its completion is counted
// in bytes on that CTA's mbarrier.
__device__ __forceinline__ void st_async_v4(uint32_t cluster_addr, float a, float b, float c, float d,
                                            uint32_t cluster_bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     cluster_addr),
                 "f"(a), "f"(b), "f"(c), "f"(d), "r"(cluster_bar)
                 : "memory");
}

// 16-byte global -> shared copy that bypasses registers (completion by group).
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit_wait_all()
{
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ float4 ld_shared_v4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// All threads of all CTAs of the cluster.
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Non-blocking probe: no suspension, the barrier's state as it is now.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *m)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                            int32_t x, int32_t y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                            int32_t x, int32_t y, int32_t z)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y), "r"(z)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap *m, uint32_t cluster_bar,
                                                 int32_t x, int32_t y, int32_t z)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(cluster_bar), "r"(x), "r"(y), "r"(z)
        : "memory");
}

// Load into this CTA's shared memory, completing bytes on the barrier of the
// pair's leader (a shared::cluster address): the second CTA of a CTA pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *m, uint32_t cluster_bar,
                                                 int32_t x, int32_t y)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(cluster_bar), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap *m, uint32_t src, int32_t x,
                                             int32_t y)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(m)),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}
__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v)
{
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v)
{
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// One lane of a converged warp (elect.sync); true in exactly that lane.
__device__ __forceinline__ bool elect_one()
{
    uint32_t pred = 0;
    asm volatile(
        "{\n\t.reg .b32 rx;\n\t.reg .pred px;\n\t"
        "elect.sync rx|px, %1;\n\t"
        "selp.u32 %0, 1, 0, px;\n\t}"
        : "=r"(pred)
        : "r"(0xFFFFFFFFu));
    return pred != 0;
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// OR of `pred` over the `count` threads that meet at named barrier `id`.
__device__ __forceinline__ bool named_bar_any(uint32_t id, uint32_t count, bool pred)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// --- tcgen05 -----------------------------------------------------------------

// TMEM management.  With a CTA pair (CG = 2) one warp of each CTA of the pair
// executes the instruction, and the columns are allocated in both.
template <int CG>
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    if constexpr (CG == 2)
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                     "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                     "r"(ncols)
                     : "memory");
}
template <int CG>
__device__ __forceinline__ void tmem_relinquish()
{
    if constexpr (CG == 2) asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    else asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
template <int CG>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    if constexpr (CG == 2)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                     : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void umma_commit_one(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Pair MMAs: the completion arrives on the barrier at the same offset in both
// CTAs of the pair (`mask`: the pair's two bits of the cluster).
__device__ __forceinline__ void umma_commit_pair(uint32_t bar, uint16_t mask)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"(mask)
        : "memory");
}

// Completion of this thread's prior MMAs arrives on `bar` (in both CTAs of a
// pair, whose cluster bits are `pair_mask`).
template <int CG>
__device__ __forceinline__ void umma_commit(uint32_t bar, uint16_t pair_mask)
{
    if constexpr (CG == 2) umma_commit_pair(bar, pair_mask);
    else umma_commit_one(bar);
}

// D[tmem] (+)= A[smem] · B[smem]; kind::f16 reads bf16, kind::tf32 reads fp32 as
// tf32, kind::f8f6f4 reads FP8 E4M3 (DT = 2).  Every kind consumes 32 bytes of K
// per MMA.
// CG = 2: one 256-row MMA over a CTA pair, issued by the pair's leader; each CTA
// supplies 128 rows of A and half of B's columns from its own shared memory (at
// the descriptors' offsets) and receives its 128 rows of D in its own TMEM.
template <int DT, int CG>
__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                     uint32_t accumulate)
{
    if constexpr (CG == 2) {
        if constexpr (DT == 0)
            asm volatile(
                "{\n\t.reg .pred p;\n\t"
                "setp.ne.b32 p, %4, 0;\n\t"
                "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
                : "memory");
        else if constexpr (DT == 2)
            asm volatile(
                "{\n\t.reg .pred p;\n\t"
                "setp.ne.b32 p, %4, 0;\n\t"
                "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
                : "memory");
        else
            asm volatile(
                "{\n\t.reg .pred p;\n\t"
                "setp.ne.b32 p, %4, 0;\n\t"
                "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
                : "memory");
    } else if constexpr (DT == 0) {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
            : "memory");
    } else if constexpr (DT == 2) {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
            : "memory");
    }
}

// Block-scaled FP8 (kind::mxf8f6f4, one E8M0 scale per 32 elements of K):
// D[tmem] (+)= (A·2^sa)·(B·2^sb).  The scales live in TMEM: row m of A reads
// lane m, column sfa + m/32; column n of B reads lane n%32 of every lane
// quarter, column sfb + n/32; the byte within the 32-bit word is the scale-ID
// field of idesc (A: bits 29-30, B: bits 4-5), which names the 32-element block
// of K that this MMA covers among the four a word holds.
// CG = 2 (a CTA pair, issued by the leader): each CTA's rows read their A
// scales, and every column its B scale, from that CTA's own TMEM in the same
// layout, so both CTAs hold all of the tile's B scales.
template <int CG>
__device__ __forceinline__ void umma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate)
{
    if constexpr (CG == 2)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
                d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %6, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
                d_tmem),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
            : "memory");
}

// Copy 32 rows x 16 bytes of shared memory into TMEM, the same 32 rows into
// each of the four lane quarters (row r -> lane 32q + r, 4 columns); issued
// by the MMA thread, in order with its MMAs.  CG = 2: issued by the pair's
// leader, each CTA's block goes into that CTA's own TMEM.
template <int CG>
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc)
{
    if constexpr (CG == 2)
        asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
    else
        asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// Descriptor of a 32-row x 16-byte block in shared memory, no swizzle: four
// 8-row core matrices of 128 contiguous bytes, 128 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_rows16(uint32_t addr)
{
    uint64_t d = (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(128u >> 4) << 16;
    d |= (uint64_t)(128u >> 4) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// Shared-memory matrix descriptor, 128-byte swizzle: start address, leading
// byte offset (MN-major: distance between 128-byte-wide column blocks; unused
// for K-major), stride byte offset 1024 (distance between 8-row groups), the
// descriptor-version bit of the sm_100 family, swizzle mode 2 (128 B).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo)
{
    uint64_t d = (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((1024u >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

#define GEMM_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), \
                   "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define GEMM_P8(i) "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), "+r"(r[i + 4]), \
                   "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7])

// 32 lanes x 32 columns of fp32 from TMEM; each thread gets its lane's row.
__device__ __forceinline__ void tmem_ld_32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
        "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
        "%30, %31}, [%32];"
        : GEMM_R8(0), GEMM_R8(8), GEMM_R8(16), GEMM_R8(24)
        : "r"(taddr));
    // The wait names the registers so no use of them is scheduled above it.
    asm volatile("tcgen05.wait::ld.sync.aligned;" : GEMM_P8(0), GEMM_P8(8), GEMM_P8(16), GEMM_P8(24)::"memory");
}

__device__ __forceinline__ void tmem_ld_16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
        "%12, %13, %14, %15}, [%16];"
        : GEMM_R8(0), GEMM_R8(8)
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" : GEMM_P8(0), GEMM_P8(8)::"memory");
}

template <int CH>
__device__ __forceinline__ void tmem_load_chunk(uint32_t taddr, float (&v)[CH])
{
    if constexpr (CH == 32) {
        uint32_t r[32];
        tmem_ld_32(taddr, r);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
    } else {
        uint32_t r[16];
        tmem_ld_16(taddr, r);
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
    }
}

// ---------------------------------------------------------------------------
// Bounded waits
// ---------------------------------------------------------------------------

struct WaitCtl {
    volatile int32_t *abort;
    int32_t *status;
    int64_t timeout_ns;
};

// Slow path of a wait: polls with a bound measured in SM clock cycles
// (clock64 is a cheap register read; the cycle budget assumes the highest SM
// clock, so at lower clocks the wall-clock bound only grows).
__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, const WaitCtl &c, int32_t site,
                                       bool heed_abort, int64_t limit_ns)
{
    const long long limit_cycles = (long long)((double)limit_ns * 2.2);
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (heed_abort && *c.abort) return false;
            if (clock64() - t0 > limit_cycles) {
                *c.abort = 1;
                atomicCAS(c.status, 0, site);
                return false;
            }
        }
    }
}

// Fast path: a short burst of non-blocking probes with no timer or flag
// reads.  (A try_wait was measured to hold the thread about 0.9 us even on a
// phase that had already completed, e.g. the first wait on a fresh barrier.)
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const WaitCtl &c, int32_t site)
{
#pragma unroll 1
    for (int i = 0; i < 256; ++i)
        if (mbar_test_wait(bar, parity)) return true;
    return wait_slow(bar, parity, c, site, true, c.timeout_ns);
}

// Bounded wait on a barrier completed from other CTAs of the cluster.
__device__ __noinline__ bool wait_bar_cluster(uint32_t bar, uint32_t parity, const WaitCtl &c, int32_t site)
{
    const long long limit_cycles = (long long)((double)c.timeout_ns * 2.2);
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*c.abort) return false;
            if (clock64() - t0 > limit_cycles) {
                *c.abort = 1;
                atomicCAS(c.status, 0, site);
                return false;
            }
        }
    }
}

// Adds with acquire-release semantics at GPU scope; returns the count before.
// The release publishes this CTA's earlier global writes (ordered before this
// thread by a CTA barrier) with the increment; the acquire makes the writes
// published by earlier increments visible (passed on by the next CTA barrier).
__device__ __forceinline__ int32_t atom_acq_rel_gpu_add(int32_t *ptr, int32_t v)
{
    int32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(ptr), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ uint64_t atom_acq_rel_gpu_add_u64(uint64_t *ptr, uint64_t v)
{
    uint64_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;" : "=l"(old) : "l"(ptr), "l"(v) : "memory");
    return old;
}

__device__ __forceinline__ uint64_t ld_acquire_gpu_u64(const uint64_t *ptr)
{
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(ptr) : "memory");
    return v;
}

// Split-K share counts: every launch adds exactly S arrivals to each share's
// count (they only grow), so a count read before this slice's own arrival lies
// in [base, base + S - 1] with base a multiple of S.  True once the other S - 1
// slices have arrived (acquire: their partials are then visible), false when
// `limit` SM cycles or the CTA's abort flag end the wait first.  Never an
// error: the slices of a one-wave launch normally arrive within a microsecond
// or two of each other, and a slice that is not resident (its SM held by
// another kernel) only makes the owner hand its share over, to be finalised
// by whichever slice arrives last.
__device__ __noinline__ bool poll_share(const uint64_t *ptr, uint32_t S, const WaitCtl &c, long long limit)
{
    uint64_t v = ld_acquire_gpu_u64(ptr);
    const uint64_t target = v - v % S + (S - 1);
    if (v >= target) return true;
    if (limit <= 0) return false;
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        __nanosleep(32);
        if (ld_acquire_gpu_u64(ptr) >= target) return true;
        if ((it & 15u) == 0 && (*c.abort || clock64() - t0 > limit)) return false;
    }
}

// Teardown waits (copies / MMAs already issued): one second, abort flag ignored.
__device__ __forceinline__ bool wait_teardown(uint32_t bar, uint32_t parity, const WaitCtl &c)
{
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, c, SITE_TEARDOWN, false, 1000000000LL);
}

// ---------------------------------------------------------------------------
// Epilogue helpers
// ---------------------------------------------------------------------------

template <int DT>
struct Elt;
template <>
struct Elt<0> {
    static constexpr int BYTES = 2;
};
template <>
struct Elt<1> {
    static constexpr int BYTES = 4;
};
template <>
struct Elt<2> {   // FP8 E4M3
    static constexpr int BYTES = 1;
};
template <>
struct Elt<3> {   // block-scaled FP8 E4M3 (MX)
    static constexpr int BYTES = 1;
};

// erfc(z) for z >= 0 by Abramowitz & Stegun, "Handbook of Mathematical
// Functions" (1964), formula 7.1.28: erf(z) = 1 - 1/(1 + a1 z + ... + a6 z^6)^16
// with absolute error at most 3e-7.  One reciprocal (the rational form of
// 7.1.26 needs a reciprocal and an exponential), six FMAs and four squarings;
// branch-free, so the 32 values of a chunk are computed side by side.  In fp32
// the sixteenth power carries the polynomial's rounding sixteen-fold: q is
// within about 1e-5 relative of erfc, far below a bf16 rounding step.
__device__ __forceinline__ float gelu_erf(float x)
{
    const float z = fabsf(x) * 0.70710678118654752440f;
    float d = fmaf(z, 0.0000430638f, 0.0002765672f);
    d = fmaf(d, z, 0.0001520143f);
    d = fmaf(d, z, 0.0092705272f);
    d = fmaf(d, z, 0.0422820123f);
    d = fmaf(d, z, 0.0705230784f);
    d = fmaf(d, z, 1.0f);
    d *= d;
    d *= d;
    d *= d;
    d *= d;   // (1 + a1 z + ... + a6 z^6)^16; infinite for large z, and then q = 0
    // q = erfc(|x|/√2); 1 + erf(x/√2) is 2 - q for x >= 0 and q for x < 0
    // (taking q directly avoids cancellation in the negative tail).
    const float q = __fdividef(1.0f, d);
    return 0.5f * x * (x >= 0.0f ? 2.0f - q : q);
}

// Applies bias (one value per column, held by lane j for column j of the
// chunk) and the activation to a 32-column row chunk.
__device__ __forceinline__ void bias_act_rows(float (&v)[32], float lane_bias, int epi, float alpha)
{
    if (alpha != 1.0f) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= alpha;
    }
    if (epi == 0) return;
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] += __shfl_sync(0xFFFFFFFFu, lane_bias, j);
    if (epi == 2) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = fmaxf(v[j], 0.0f);
    } else if (epi == 3) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = gelu_erf(v[j]);
    }
}

// Gated (GLU-style) epilogue of a 32-column output chunk: g holds the gate
// chunk, u the up chunk of the fused accumulator (one row per lane); lane j
// holds column j's biases.  g becomes act(alpha·g + b_gate) · (alpha·u + b_up),
// act ReLU (epi 7), GELU (8) or SiLU x / (1 + e^-x) (9).
__device__ __forceinline__ void glu_rows(float (&g)[32], const float (&u)[32], float gate_bias, float up_bias, int epi,
                                         float alpha)
{
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        float x = g[j], y = u[j];
        if (alpha != 1.0f) {
            x *= alpha;
            y *= alpha;
        }
        x += __shfl_sync(0xFFFFFFFFu, gate_bias, j);
        y += __shfl_sync(0xFFFFFFFFu, up_bias, j);
        const float a = epi == 7 ? fmaxf(x, 0.0f) : epi == 8 ? gelu_erf(x) : __fdividef(x, 1.0f + __expf(-x));
        g[j] = a * y;
    }
}

__device__ __forceinline__ void bias_act_cols(float (&v)[16], float row_bias, int epi, float alpha)
{
    if (alpha != 1.0f) {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] *= alpha;
    }
    if (epi == 0) return;
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] += row_bias;
    if (epi == 2) {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = fmaxf(v[j], 0.0f);
    } else if (epi == 3) {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = gelu_erf(v[j]);
    }
}

// Residual: R is the caller's [M, N] row-major tensor of C's type (it may be C
// itself: each element is read once, before its own store).  Unswapped, a
// thread holds 32 columns n0.. of row m; swapped, 16 rows m0.. of column n.
template <int DT>
__device__ __forceinline__ void add_residual_rows(float (&v)[32], const void *R, int64_t ld, int32_t m, int32_t n0,
                                                  int32_t M, int32_t N)
{
    if (m >= M) return;
    if constexpr (DT == 0) {
        const uint16_t *row = static_cast<const uint16_t *>(R) + (size_t)m * (size_t)ld + n0;
        if (n0 + 32 <= N) {
            const uint4 *p4 = reinterpret_cast<const uint4 *>(row);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 q = p4[i];
                const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    v[8 * i + 2 * k] += __uint_as_float(w[k] << 16);
                    v[8 * i + 2 * k + 1] += __uint_as_float(w[k] & 0xFFFF0000u);
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (n0 + j < N) v[j] += __uint_as_float((uint32_t)row[j] << 16);
        }
    } else {
        const float *row = static_cast<const float *>(R) + (size_t)m * (size_t)ld + n0;
        if (n0 + 32 <= N) {
            const float4 *p4 = reinterpret_cast<const float4 *>(row);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 q = p4[i];
                v[4 * i] += q.x;
                v[4 * i + 1] += q.y;
                v[4 * i + 2] += q.z;
                v[4 * i + 3] += q.w;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (n0 + j < N) v[j] += row[j];
        }
    }
}

template <int DT>
__device__ __forceinline__ void add_residual_cols(float (&v)[16], const void *R, int64_t ld, int32_t m0, int32_t n,
                                                  int32_t M, int32_t N)
{
    if (n >= N) return;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        if (m0 + j < M) {
            const size_t at = (size_t)(m0 + j) * (size_t)ld + n;
            if constexpr (DT == 0) v[j] += __uint_as_float((uint32_t)static_cast<const uint16_t *>(R)[at] << 16);
            else v[j] += static_cast<const float *>(R)[at];
        }
    }
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16)
{
    return __uint_as_float(bits16 << 16);
}

template <int DT>
__device__ __forceinline__ float load_bias1(const void *bias, int n, int limit)
{
    if (n >= limit) return 0.0f;
    if constexpr (DT == 0) return bf16_bits_to_float(__ldg(reinterpret_cast<const uint16_t *>(bias) + n));
    else return __ldg(reinterpret_cast<const float *>(bias) + n);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Per-warp store state: two staging buffers used alternately.
struct StoreRing {
    uint32_t buf0;      // shared address of this warp's first staging buffer
    uint32_t buf_bytes;
    uint32_t count;     // chunks issued so far
};

// Unswapped store: the warp's 32 rows (one per lane) x 32 columns -> staging
// (swizzled like the tensor map) -> one TMA store of a 32x32 box at (x, y).
template <int DT>
__device__ __forceinline__ void store_rows_chunk(const CUtensorMap *tmC, StoreRing &ring, const float (&v)[32],
                                                 int lane, int x, int y, bool in_bounds)
{
    const uint32_t buf = ring.buf0 + (ring.count & 1u) * ring.buf_bytes;
    if (lane == 0) bulk_wait_read_1();
    __syncwarp();
    if constexpr (DT == 0) {
        // 64-byte rows, 64-byte swizzle: 16-byte chunk i of row r lands at i ^ ((r >> 1) & 3)
        const uint32_t row = buf + (uint32_t)lane * 64u;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t phys = (uint32_t)(i ^ ((lane >> 1) & 3)) * 16u;
            st_shared_v4(row + phys, pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                         pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
        }
    } else {
        // 128-byte rows, 128-byte swizzle: chunk i of row r lands at i ^ (r & 7)
        const uint32_t row = buf + (uint32_t)lane * 128u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t phys = (uint32_t)(i ^ (lane & 7)) * 16u;
            st_shared_v4(row + phys, __float_as_uint(v[4 * i]), __float_as_uint(v[4 * i + 1]),
                         __float_as_uint(v[4 * i + 2]), __float_as_uint(v[4 * i + 3]));
        }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && in_bounds) {
        tma_store_2d(tmC, buf, x, y);
        bulk_commit();
    }
    ring.count++;
}

// Swapped store: lane = output column n, 16 values = 16 output rows m.
// Staging is [16 rows][32 columns] (no swizzle); one TMA store of a 32x16 box.
template <int DT>
__device__ __forceinline__ void store_cols_chunk(const CUtensorMap *tmC, StoreRing &ring, const float (&v)[16],
                                                 int lane, int x, int y, bool in_bounds)
{
    const uint32_t buf = ring.buf0 + (ring.count & 1u) * ring.buf_bytes;
    if (lane == 0) bulk_wait_read_1();
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        if constexpr (DT == 0) {
            const __nv_bfloat16 h = __float2bfloat16_rn(v[j]);
            st_shared_u16(buf + (uint32_t)(j * 64 + lane * 2), *reinterpret_cast<const uint16_t *>(&h));
        } else {
            st_shared_u32(buf + (uint32_t)(j * 128 + lane * 4), __float_as_uint(v[j]));
        }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && in_bounds) {
        tma_store_2d(tmC, buf, x, y);
        bulk_commit();
    }
    ring.count++;
}

// One pipeline stage's MMAs: KSTEPS K-steps of 32 bytes, each as HALVES
// 128-row MMAs into consecutive accumulator column blocks.
struct MmaStage {
    uint32_t d0;            // TMEM address of the accumulator
    uint64_t adesc, bdesc;  // descriptors of the stage's A and B tiles
    uint32_t idesc;
    uint32_t a_span_step, b_span_step, a_half_step;  // 16-byte units
    uint32_t bn;
    bool accumulate_first;  // false on the unit's first K-block
};

template <int DT, bool A_MN, bool B_MN, int KSTEPS, int HALVES, int CG = 1>
__device__ __forceinline__ void issue_stage(const MmaStage &st)
{
    constexpr int ELT = Elt<DT>::BYTES;
    constexpr uint32_t MN_KSTEP16 = ((32u / ELT) * 128u) >> 4;
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
        const uint32_t a_k = A_MN ? (uint32_t)kk * MN_KSTEP16 : (uint32_t)(kk >> 2) * st.a_span_step + (kk & 3) * 2u;
        const uint32_t b_k = B_MN ? (uint32_t)kk * MN_KSTEP16 : (uint32_t)(kk >> 2) * st.b_span_step + (kk & 3) * 2u;
        const uint32_t acc = (st.accumulate_first || kk != 0) ? 1u : 0u;
#pragma unroll
        for (int h = 0; h < HALVES; ++h)
            umma<DT, CG>(st.d0 + (uint32_t)h * st.bn, st.adesc + a_k + (uint32_t)h * st.a_half_step,
                         st.bdesc + b_k, st.idesc, acc);
    }
}

// One block-scaled (MX) stage: first the stage's scale atoms go from shared
// memory to its TMEM slot (A's atoms [half][K atom] at columns (h·KA + a)·4,
// then B's at (HALVES·KA + a·bn_atoms + j)·4 so that a K atom's B columns are
// contiguous, n/32 apart), then the MMAs, each naming its 32-element block of
// K by the scale ID (kk mod 4) and its atom by the slot column (kk / 4).
template <bool A_MN, bool B_MN, int KSTEPS, int HALVES, int CG = 1>
__device__ __forceinline__ void issue_stage_mx(const MmaStage &st, uint32_t slot, uint32_t sf_smem, int bn_atoms)
{
    constexpr int KA = KSTEPS / 4;
    constexpr uint32_t MN_KSTEP16 = (32u * 128u) >> 4;
#pragma unroll
    for (int h = 0; h < HALVES; ++h)
#pragma unroll
        for (int a = 0; a < KA; ++a)
            tmem_cp_32x128b_x4<CG>(slot + (uint32_t)(h * KA + a) * 4u,
                               smem_desc_rows16(sf_smem + (uint32_t)(h * KA + a) * 512u));
    for (int j = 0; j < bn_atoms; ++j)
#pragma unroll
        for (int a = 0; a < KA; ++a)
            tmem_cp_32x128b_x4<CG>(slot + (uint32_t)(HALVES * KA + a * bn_atoms + j) * 4u,
                               smem_desc_rows16(sf_smem + (uint32_t)(HALVES * KA + j * KA + a) * 512u));
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
        const uint32_t a_k = A_MN ? (uint32_t)kk * MN_KSTEP16 : (uint32_t)(kk >> 2) * st.a_span_step + (kk & 3) * 2u;
        const uint32_t b_k = B_MN ? (uint32_t)kk * MN_KSTEP16 : (uint32_t)(kk >> 2) * st.b_span_step + (kk & 3) * 2u;
        const uint32_t acc = (st.accumulate_first || kk != 0) ? 1u : 0u;
        const uint32_t id = st.idesc | ((uint32_t)(kk & 3) << 29) | ((uint32_t)(kk & 3) << 4);
        const uint32_t sfb = slot + (uint32_t)(HALVES * KA + (kk >> 2) * bn_atoms) * 4u;
#pragma unroll
        for (int h = 0; h < HALVES; ++h)
            umma_mx<CG>(st.d0 + (uint32_t)h * st.bn, st.adesc + a_k + (uint32_t)h * st.a_half_step, st.bdesc + b_k, id,
                    slot + (uint32_t)(h * KA + (kk >> 2)) * 4u, sfb, acc);
    }
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------

template <int DT, bool A_MN, bool B_MN, int CG>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tcgen05_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmSA,
                        const __grid_constant__ CUtensorMap tmSB, const KernelParams p)
{
    constexpr int ELT = Elt<DT>::BYTES;
    constexpr int ODT = DT >= 2 ? 0 : DT;            // type of C, bias and R (FP8 operands give bf16)
    constexpr int SPAN = 128 / ELT;                  // elements in one 128-byte swizzle span

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const gbase = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // CTA pair (cta_group::2): consecutive CTAs form a cluster of two; rank 0
    // (the leader) issues the MMAs for both, each CTA holds 128 rows of the
    // tile.  Both walk the same units.
    constexpr bool pair = CG == 2;
    const uint32_t prank = pair ? (blockIdx.x & 1u) : 0u;
    // A pair is two consecutive ranks of its cluster: of two CTAs, or, when the
    // K slices of a pair tile also form one cluster, of 2 x S.
    const uint32_t crank = (pair || p.cluster_k > 1) ? cluster_ctarank() : 0u;
    const uint32_t lead_rank = crank & ~1u;
    const uint16_t pair_mask = (uint16_t)(3u << lead_rank);
    const int64_t unit0 = pair ? (int64_t)(blockIdx.x >> 1) : (int64_t)blockIdx.x;
    const int64_t unit_step = pair ? (int64_t)(gridDim.x >> 1) : (int64_t)gridDim.x;
    const int32_t cta_rows = pair ? 128 : p.bm;        // tile rows held by this CTA
    const int32_t cta_bcols = pair ? p.bn / 2 : p.bn;  // B columns loaded by this CTA

    const uint32_t bars = base + p.off_bar;
    const uint32_t full0 = bars;
    const uint32_t empty0 = bars + 8u * (uint32_t)p.stages;
    const uint32_t tfull0 = bars + 16u * (uint32_t)p.stages;
    const uint32_t tempty0 = tfull0 + 16u;
    const uint32_t teardown_bar = tfull0 + 32u;
    const uint32_t never_bar = tfull0 + 40u;
    const uint32_t tmem_slot = tfull0 + 48u;
    const uint32_t peer_ready_bar = tfull0 + 64u;   // cluster split-K: the other slices' rings are free
    const uint32_t recv_bar = tfull0 + 72u;         // cluster split-K: every partial for my blocks has landed
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(gbase + (tmem_slot - base) + 4);
    volatile int32_t *last_flag = reinterpret_cast<volatile int32_t *>(gbase + (tmem_slot - base) + 8);

    // The tensor maps are this launch's own parameters: fetching them into the
    // TMA unit's descriptor cache may start at once, ahead of the wait on the
    // previous kernel below, instead of stalling the first copy.
    // The same for the parameter block: its first reads miss the constant
    // cache (measured: the first schedule lookup took about 0.8 us), so one
    // thread touches every part of it now, while the previous kernel drains.
    if (threadIdx.x == 32) {
        if (p.num_kb > 0) {
            prefetch_tmap(&tmA);
            prefetch_tmap(&tmB);
            if constexpr (DT == 3) {
                prefetch_tmap(&tmSA);
                prefetch_tmap(&tmSB);
            }
        }
        prefetch_tmap(&tmC);
        asm volatile("" ::"r"(p.rows), "r"(p.num_units), "r"(p.tiles_m), "r"(p.staging_buf_bytes), "l"(p.bias),
                     "l"(p.status), "r"(p.cluster_k), "r"(p.off_staging), "l"(p.workspace));
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(full0 + 8u * s, pair ? 2u : 1u);   // pair: both producers arrive on the leader's
            mbar_init(empty0 + 8u * s, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(tfull0 + 8u * i, 1);
            mbar_init(tempty0 + 8u * i, pair ? 2u : (uint32_t)kEpiThreads);  // pair: one arrival per CTA
        }
        mbar_init(teardown_bar, 1);
        mbar_init(never_bar, 1);
        if (p.cluster_k > 1) {
            mbar_init(peer_ready_bar, (uint32_t)(p.cluster_k - 1));
            mbar_init(recv_bar, 1);
        }
        *abort_flag = 0;
        *last_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc<CG>(tmem_slot, p.tmem_cols);
        tmem_relinquish<CG>();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t *>(gbase + (tmem_slot - base));
    // Peers arrive on this CTA's barriers: none may do so before every CTA of
    // the cluster has initialised its own.
    if (p.cluster_k > 1 || pair) cluster_sync_all();
    // Programmatic dependent launch: the set-up above may overlap the previous
    // kernel on the stream; global memory is touched only once that kernel has
    // finished and its writes are visible.  The next kernel may then begin its
    // own set-up as soon as SMs free up.
    // The epilogue warps, which read bias and R and write C, the split-K
    // workspace, the counters and the status word, wait here, and so does the
    // MMA warp, so that its bounded waits start only once the previous kernel
    // has finished.  The producer waits right before its first copy: its
    // schedule and barrier work before that (whose first pass fetches cold
    // code and parameters, measured at about 0.9 us) overlaps the previous
    // kernel's drain.  Operands declared independent of the previous kernel
    // (early mask: bit 0 MMA-A, bit 1 MMA-B) let the producer go further: with
    // one it copies that operand's first stages before waiting; with both
    // neither it nor the MMA warp waits.
    const uint32_t early_mask = (uint32_t)p.early_mask & 3u;
    if (warp >= 2 || (warp == 1 && early_mask != 3u)) asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    WaitCtl ctl{abort_flag, p.status, p.timeout_ns};

    // Roles run warp-converged: every lane walks the same schedule (so the
    // loop state is warp-uniform), one elected lane issues the TMA copies and
    // the MMAs, and the wait outcome is agreed with a warp vote.
    if (warp == 0) {
        // ------------------------------------------------------------------
        // TMA producer
        // ------------------------------------------------------------------
        const bool leader = elect_one();
        const int32_t stages = p.stages, bm = p.bm, bn = p.bn, bk = p.bk;
        const uint32_t a_bytes = p.a_stage_bytes, b_bytes = p.b_stage_bytes, tx = p.tx_bytes;
        const uint32_t sb0 = base + p.off_b;
        const int32_t a_loads = A_MN ? cta_rows / SPAN : bk / SPAN;
        const int32_t b_loads = B_MN ? cta_bcols / SPAN : bk / SPAN;
        const bool a3d = p.a_span3d != 0, b3d = p.b_span3d != 0;
        // One stage's copies, split by operand: bit 0 of `what` issues MMA-A's
        // panel (with its MX scale atoms), bit 1 MMA-B's; `arm` first posts the
        // stage's full byte count on its barrier.
        auto fill = [&](uint32_t stage, const SchedUnit &w, int32_t kb, uint32_t what, bool arm) {
            const int32_t ra = w.tile_m * bm + (int32_t)prank * 128;
            const int32_t rb = w.tile_n * bn + (int32_t)prank * cta_bcols;
            const uint32_t fb = full0 + 8u * stage;
            const uint32_t sa = base + stage * a_bytes;
            const uint32_t sb = sb0 + stage * b_bytes;
            const int32_t k0 = kb * bk;
            if (leader && prank == 0) {
                if (arm) mbar_arrive_expect_tx(fb, tx);
                // K-major operand: boxes of [rows x one span of K], one per span;
                // MN-major operand: boxes of [bk x one span of MN], one per span.
                // A 3-D view takes all of the stage's spans in one copy; the
                // boxes land span after span, as the per-span copies would.
                if (what & 1u) {
                    if (a3d) {
                        if constexpr (A_MN) tma_load_3d(sa, &tmA, fb, 0, k0, ra / SPAN);
                        else tma_load_3d(sa, &tmA, fb, 0, ra, k0 / SPAN);
                    } else {
                        for (int32_t j = 0; j < a_loads; ++j) {
                            if constexpr (A_MN) tma_load_2d(sa + (uint32_t)(j * bk * 128), &tmA, fb, ra + j * SPAN, k0);
                            else tma_load_2d(sa + (uint32_t)(j * cta_rows * 128), &tmA, fb, k0 + j * SPAN, ra);
                        }
                    }
                }
                if (what & 2u) {
                    if (b3d) {
                        if constexpr (B_MN) tma_load_3d(sb, &tmB, fb, 0, k0, rb / SPAN);
                        else tma_load_3d(sb, &tmB, fb, 0, rb, k0 / SPAN);
                    } else {
                        for (int32_t j = 0; j < b_loads; ++j) {
                            if constexpr (B_MN) tma_load_2d(sb + (uint32_t)(j * bk * 128), &tmB, fb, rb + j * SPAN, k0);
                            else tma_load_2d(sb + (uint32_t)(j * cta_bcols * 128), &tmB, fb, k0 + j * SPAN, rb);
                        }
                    }
                }
                if constexpr (DT == 3) {
                    // The stage's scale atoms, one tensor copy per operand (the
                    // packed array seen as [row atoms][K atoms][128 words]):
                    // for the tile's 128-row groups of MMA-A, then its 128-column
                    // groups of MMA-B (one atom when bn < 128: such a tile
                    // starts on an atom), their bk/128 consecutive K atoms,
                    // landing as [group][K atom] atoms of 512 bytes.  Swapped,
                    // MMA-A is B (rows along N) and MMA-B is A.
                    const uint32_t ka = (uint32_t)bk / 128u, run = ka * 512u;
                    const uint32_t sf = base + p.off_sf + stage * p.sf_stage_bytes;
                    const int32_t k_atom = kb * (int32_t)ka;
                    const CUtensorMap *sm_a = A_MN || p.swap_ab ? &tmSB : &tmSA;
                    const CUtensorMap *sm_b = A_MN || p.swap_ab ? &tmSA : &tmSB;
                    const int32_t na = pair ? 1 : bm / 128;
                    if (what & 1u) tma_load_3d(sf, sm_a, fb, 0, k_atom, w.tile_m * (bm / 128));
                    if (what & 2u) tma_load_3d(sf + (uint32_t)na * run, sm_b, fb, 0, k_atom, w.tile_n * bn / 128);
                }
            } else if (leader) {
                if constexpr (pair) {
                    // Second CTA of a pair: its halves land in its own shared
                    // memory and complete on the leader's barrier, where the MMAs wait.
                    const uint32_t fbr = mapa_u32(fb, lead_rank);
                    if (arm) mbar_arrive_expect_tx_remote(fbr, tx);
                    if (what & 1u) {
                        if (a3d) {
                            if constexpr (A_MN) tma_load_3d_pair(sa, &tmA, fbr, 0, k0, ra / SPAN);
                            else tma_load_3d_pair(sa, &tmA, fbr, 0, ra, k0 / SPAN);
                        } else {
                            for (int32_t j = 0; j < a_loads; ++j) {
                                if constexpr (A_MN)
                                    tma_load_2d_pair(sa + (uint32_t)(j * bk * 128), &tmA, fbr, ra + j * SPAN, k0);
                                else
                                    tma_load_2d_pair(sa + (uint32_t)(j * cta_rows * 128), &tmA, fbr, k0 + j * SPAN,
                                                     ra);
                            }
                        }
                    }
                    if (what & 2u) {
                        if (b3d) {
                            if constexpr (B_MN) tma_load_3d_pair(sb, &tmB, fbr, 0, k0, rb / SPAN);
                            else tma_load_3d_pair(sb, &tmB, fbr, 0, rb, k0 / SPAN);
                        } else {
                            for (int32_t j = 0; j < b_loads; ++j) {
                                if constexpr (B_MN)
                                    tma_load_2d_pair(sb + (uint32_t)(j * bk * 128), &tmB, fbr, rb + j * SPAN, k0);
                                else
                                    tma_load_2d_pair(sb + (uint32_t)(j * cta_bcols * 128), &tmB, fbr,
                                                     k0 + j * SPAN, rb);
                            }
                        }
                    }
                    if constexpr (DT == 3) {
                        // MX: this CTA's 128 rows of A scales and all of the
                        // tile's B scales (the pair MMA reads each CTA's own).
                        const uint32_t ka = (uint32_t)bk / 128u, run = ka * 512u;
                        const uint32_t sf = base + p.off_sf + stage * p.sf_stage_bytes;
                        const int32_t k_atom = kb * (int32_t)ka;
                        if (what & 1u) tma_load_3d_pair(sf, &tmSA, fbr, 0, k_atom, w.tile_m * 2 + 1);
                        if (what & 2u) tma_load_3d_pair(sf + run, &tmSB, fbr, 0, k_atom, w.tile_n * bn / 128);
                    }
                }
            }
            __syncwarp();
        };

        uint32_t stage = 0, phase = 0, armed = 0, armed_parity = 0;
        // One operand declared independent of the previous kernel (early mask
        // 1 or 2): its copies for the first pass over the ring go out before
        // the dependency wait (the ring is fresh, so no slot needs waiting
        // for), and the other operand's follow once the previous kernel's
        // writes are visible.
        int32_t pre = 0;
        bool waited = early_mask == 3u;
        if (early_mask == 1u || early_mask == 2u) {
            for (int64_t u = unit0; pre < stages && u < p.num_units; u += unit_step) {
                const SchedUnit w = schedule_unit(u, p.tiles_m, p.tiles_n, p.split_k, p.raster, p.group, p.num_kb);
                for (int32_t kb = w.kb_begin; pre < stages && kb < w.kb_end; ++kb, ++pre)
                    fill((uint32_t)pre, w, kb, early_mask, true);
            }
            asm volatile("griddepcontrol.wait;" ::: "memory");
            waited = true;
        }
        bool ok = true;
        int32_t filled = 0;
        for (int64_t u = unit0; ok && u < p.num_units; u += unit_step) {
            const SchedUnit w = schedule_unit(u, p.tiles_m, p.tiles_n, p.split_k, p.raster, p.group, p.num_kb);
            for (int32_t kb = w.kb_begin; kb < w.kb_end; ++kb) {
                if (filled < pre) {
                    fill(stage, w, kb, 3u & ~early_mask, false);    // the deferred operand
                } else {
                    ok = __all_sync(0xFFFFFFFFu, wait_bar(empty0 + 8u * stage, phase ^ 1u, ctl, SITE_PRODUCER_EMPTY));
                    if (!ok) break;
                    if (!waited) {
                        asm volatile("griddepcontrol.wait;" ::: "memory");
                        waited = true;
                    }
                    fill(stage, w, kb, 3u, true);
                }
                ++filled;
                armed |= 1u << stage;
                armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == (uint32_t)stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        // Every armed stage's last copy must land before the CTA may exit.  The
        // second CTA of a pair completes its copies on the leader's barriers; the
        // leader's MMAs consume them before the pair's closing cluster barrier.
        if (prank == 0)
            for (int s = 0; s < stages; ++s)
                if ((armed >> s) & 1u) wait_teardown(full0 + 8u * s, (armed_parity >> s) & 1u, ctl);
    } else if (warp == 1) {
        // ------------------------------------------------------------------
        // MMA issuer (in a CTA pair, the leader's warp issues for both CTAs)
        // ------------------------------------------------------------------
        if (prank == 0) {
        const bool leader = elect_one();
        const int32_t stages = p.stages, bn = p.bn, bk = p.bk;
        const uint32_t a_bytes = p.a_stage_bytes, b_bytes = p.b_stage_bytes, idesc = p.idesc;
        const uint32_t sb0 = base + p.off_b, acc_cols = p.acc_cols, n_acc = p.n_acc;
        const uint32_t a_lbo = p.a_lbo, b_lbo = p.b_lbo;
        const int32_t ksteps = bk * ELT / 32;
        const int32_t halves = pair ? 1 : p.bm / 128;
        // Descriptor increments, in the 16-byte units of the start-address field:
        // next 128-row half of A; next 128-byte K span of a K-major operand.
        const uint32_t a_half_step = A_MN ? (uint32_t)((128 / SPAN) * bk * 128) >> 4 : (128u * 128u) >> 4;
        const uint32_t a_span_step = (uint32_t)(cta_rows * 128) >> 4;
        const uint32_t b_span_step = (uint32_t)(cta_bcols * 128) >> 4;
        uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
        bool issued = false, ok = true;
        for (int64_t u = unit0; ok && u < p.num_units; u += unit_step) {
            const SchedUnit w = schedule_unit(u, p.tiles_m, p.tiles_n, p.split_k, p.raster, p.group, p.num_kb);
            const int32_t nk = w.kb_end - w.kb_begin;
            // A pair's accumulator is free once both CTAs' epilogues have drained it
            // (the second arrives remotely, hence the cluster-scope wait).
            ok = __all_sync(0xFFFFFFFFu, pair ? wait_bar_cluster(tempty0 + 8u * acc, acc_phase ^ 1u, ctl,
                                                                 SITE_MMA_TMEM_EMPTY)
                                              : wait_bar(tempty0 + 8u * acc, acc_phase ^ 1u, ctl,
                                                         SITE_MMA_TMEM_EMPTY));
            if (!ok) break;
            tc_fence_after();
            const uint32_t d0 = tmem_base + acc * acc_cols;
            for (int32_t kb = 0; kb < nk; ++kb) {
                ok = __all_sync(0xFFFFFFFFu, wait_bar(full0 + 8u * stage, phase, ctl, SITE_MMA_FULL));
                if (!ok) break;
                tc_fence_after();
                const uint64_t adesc = smem_desc(base + stage * a_bytes, a_lbo);
                const uint64_t bdesc = smem_desc(sb0 + stage * b_bytes, b_lbo);
                if (leader) {
                    // The k-step loop is unrolled for every (K steps, halves) the
                    // rules allow: with a runtime bound the loop bookkeeping costs
                    // more than an MMA's issue and starves the tensor pipe.
                    const MmaStage st{d0, adesc, bdesc, idesc, a_span_step, b_span_step, a_half_step,
                                      (uint32_t)bn, kb != 0};
                    if constexpr (DT == 3) {
                        const uint32_t slot = tmem_base + p.sc_col0 + stage * p.sc_stage_cols;
                        const uint32_t sf = base + p.off_sf + stage * p.sf_stage_bytes;
                        const int bn_atoms = max(1, bn / 128);
                        if constexpr (pair) {   // one 256-row MMA per K step over both CTAs
                            if (ksteps == 4) issue_stage_mx<A_MN, B_MN, 4, 1, 2>(st, slot, sf, bn_atoms);
                            else issue_stage_mx<A_MN, B_MN, 8, 1, 2>(st, slot, sf, bn_atoms);
                        } else {
                            switch (ksteps * 2 + halves - 1) {
                            case 8: issue_stage_mx<A_MN, B_MN, 4, 1>(st, slot, sf, bn_atoms); break;
                            case 9: issue_stage_mx<A_MN, B_MN, 4, 2>(st, slot, sf, bn_atoms); break;
                            case 16: issue_stage_mx<A_MN, B_MN, 8, 1>(st, slot, sf, bn_atoms); break;
                            default: issue_stage_mx<A_MN, B_MN, 8, 2>(st, slot, sf, bn_atoms); break;
                            }
                        }
                        umma_commit<CG>(empty0 + 8u * stage, pair_mask);  // slot is free once these MMAs have read it
                    } else if constexpr (pair) {
                        switch (ksteps) {
                        case 4: issue_stage<DT, A_MN, B_MN, 4, 1, 2>(st); break;
                        case 8: issue_stage<DT, A_MN, B_MN, 8, 1, 2>(st); break;
                        case 12: issue_stage<DT, A_MN, B_MN, 12, 1, 2>(st); break;
                        default: issue_stage<DT, A_MN, B_MN, 16, 1, 2>(st); break;
                        }
                        umma_commit<CG>(empty0 + 8u * stage, pair_mask);  // both CTAs' slots are free
                    } else {
                        switch (ksteps * 2 + halves - 1) {
                        case 8: issue_stage<DT, A_MN, B_MN, 4, 1>(st); break;
                        case 9: issue_stage<DT, A_MN, B_MN, 4, 2>(st); break;
                        case 16: issue_stage<DT, A_MN, B_MN, 8, 1>(st); break;
                        case 17: issue_stage<DT, A_MN, B_MN, 8, 2>(st); break;
                        case 24: issue_stage<DT, A_MN, B_MN, 12, 1>(st); break;
                        case 25: issue_stage<DT, A_MN, B_MN, 12, 2>(st); break;
                        case 32: issue_stage<DT, A_MN, B_MN, 16, 1>(st); break;
                        default: issue_stage<DT, A_MN, B_MN, 16, 2>(st); break;
                        }
                        umma_commit<CG>(empty0 + 8u * stage, pair_mask);  // slot is free once these MMAs have read it
                    }
                }
                __syncwarp();
                issued = true;
                if (++stage == (uint32_t)stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) break;
            if (leader) {
                if (nk > 0) {
                    umma_commit<CG>(tfull0 + 8u * acc, pair_mask);
                } else {
                    mbar_arrive(tfull0 + 8u * acc);
                    if (pair) mbar_arrive_remote(mapa_u32(tfull0 + 8u * acc, lead_rank | 1u));
                }
            }
            __syncwarp();
            if (++acc == n_acc) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (issued) {
            if (leader) umma_commit<CG>(teardown_bar, pair_mask);
            __syncwarp();
            wait_teardown(teardown_bar, 0, ctl);
        }
        }
    } else {
        // ------------------------------------------------------------------
        // Epilogue: TMEM -> registers -> (+bias, act) -> staging -> TMA store.
        // Eight warps: two per TMEM sub-partition (warp % 4), splitting the
        // accumulator's column chunks between them (even / odd chunks).  The
        // bias of a unit is loaded (one value per lane and chunk) before its
        // accumulator is ready, so that load overlaps the main loop.
        // ------------------------------------------------------------------
        const int32_t e_bn = p.bn, e_bm = p.bm, e_epi = p.epi, e_cols = p.cols, e_rows = p.rows;
        const void *const e_resid = p.residual;   // C = act(A·B + bias) + R when set
        const float e_alpha = p.alpha;          // C = act(alpha·(A·B) + bias) (+ R)
        const bool e_res = e_resid != nullptr;
        const int32_t e_split_k = p.split_k, e_swap_ab = p.swap_ab;
        const bool e_coop = p.coop_fixup != 0;
        const bool e_cluster = p.cluster_k > 1;
        const uint32_t e_acc_cols = p.acc_cols, e_n_acc = p.n_acc;
        const void *const e_bias = p.bias;
        float *const e_workspace = p.workspace;
        int32_t *const e_counters = p.counters;
        uint64_t *const e_epochs = p.epochs;
        const int q = warp & 3;             // TMEM sub-partition this warp may read
        const int ew = warp - 2;            // 0..7
        const int cg = ew >> 2;             // column-chunk parity handled by this warp
        StoreRing ring{base + p.off_staging + (uint32_t)ew * 2u * p.staging_buf_bytes, p.staging_buf_bytes, 0};
        uint32_t acc = 0, acc_phase = 0;
        bool first = true;
        // Hands the drained accumulator back to the MMA issuer: every epilogue
        // thread arrives, or, in a CTA pair, the CTA's epilogue arrives once on
        // the leader's barrier.
        auto release_acc = [&](uint32_t a) {
            tc_fence_before();
            if (!pair) {
                mbar_arrive(tempty0 + 8u * a);
            } else {
                named_bar_sync(1, kEpiThreads);
                if (ew == 0 && lane == 0) {
                    if (prank == 0) mbar_arrive(tempty0 + 8u * a);
                    else mbar_arrive_remote(mapa_u32(tempty0 + 8u * a, lead_rank));
                }
            }
        };
        const int32_t halves = pair ? 1 : e_bm / 128;
        const int32_t tile_elems = cta_rows * e_bn;   // one CTA's share of a tile (split-K exchange)
        const int32_t chunks = e_swap_ab ? e_bn / 16 : e_bn / 32;
        for (int64_t u = unit0; u < p.num_units; u += unit_step) {
            const SchedUnit w = schedule_unit(u, p.tiles_m, p.tiles_n, e_split_k, p.raster, p.group, p.num_kb);
            const int32_t r0 = w.tile_m * e_bm + (int32_t)prank * 128;
            const int32_t xtile = pair ? w.tile * 2 + (int32_t)prank : w.tile;  // split-K exchange tile
            const int32_t c0 = w.tile_n * e_bn;
            // bias: unswapped, lane j holds column c0 + c*32 + j of each of this
            // warp's chunks; swapped, each lane holds its row's value per half.
            float bcol[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            float brow[2] = {0.0f, 0.0f};
            if (e_epi != 0) {
                if (!e_swap_ab) {
#pragma unroll
                    for (int ci = 0; ci < 4; ++ci) {
                        const int32_t c = cg + 2 * ci;
                        if (c < chunks) bcol[ci] = load_bias1<ODT>(e_bias, c0 + c * 32 + lane, e_cols);
                    }
                } else {
#pragma unroll
                    for (int h = 0; h < 2; ++h)
                        if (h < halves) brow[h] = load_bias1<ODT>(e_bias, r0 + h * 128 + q * 32 + lane, e_rows);
                }
            }
            bool ok = true;
            if (first && p.debug_stall) ok = wait_bar(never_bar, 0, ctl, SITE_EPI_STALL);
            first = false;
            if (ok) ok = wait_bar(tfull0 + 8u * acc, acc_phase, ctl, SITE_EPI_TMEM_FULL);
            if (named_bar_any(1, kEpiThreads, !ok)) break;
            tc_fence_after();
            const int32_t nk = w.kb_end - w.kb_begin;
            const uint32_t tacc = tmem_base + acc * e_acc_cols + ((uint32_t)(q * 32) << 16);
            if (e_cluster) {
                // Split-K inside a cluster: CTA rank s of the cluster is K slice s of
                // this tile (units are tile-major, slice fastest; one unit per CTA).
                // The tile's 128-row x 32-column blocks are dealt out in groups of
                // gsz: pairs (an even and an odd chunk, so that both warps of a
                // sub-partition get work) when there are at least two per slice,
                // else single blocks; group j belongs to slice j mod S.  Each slice pushes the
                // blocks it does not own into their owner's pipeline ring (free once
                // the owner's MMAs are done, which the owner announces), the owner
                // adds the S partials in slice order and runs the epilogue.
                // Swapped, a block is 128 rows x 16 columns (8 KB, half a slot).
                // With an area of its own (off_recv) the partials need no ring,
                // so no slice waits for another: a push may even land before
                // its owner has posted the expected bytes (the transaction count
                // goes negative for a while; the phase still needs the owner's
                // arrival).
                const int32_t S = e_split_k, me = w.split;
                const int32_t nblocks = halves * chunks;
                const int32_t gsz = nblocks >= 2 * S ? 2 : 1;
                const uint32_t blk_bytes = e_swap_ab ? kRedBlockBytes / 2u : kRedBlockBytes;
                const bool own_area = p.off_recv != 0u;
                const uint32_t rbase = own_area ? base + p.off_recv : base;
                // Slice o's CTA holding the same rows as this one (a pair tile's
                // slices are pairs 0..S-1 of the cluster).
                auto slice_rank = [&](int32_t o) { return pair ? 2u * (uint32_t)o + prank : (uint32_t)o; };
                if (ew == 0 && lane == 0) {
                    uint32_t owned = 0;
                    for (int32_t b = 0; b < nblocks; ++b) owned += ((b / gsz) % S == me) ? 1u : 0u;
                    mbar_arrive_expect_tx(recv_bar, owned * (uint32_t)(S - 1) * blk_bytes);
                    if (!own_area)
                        for (int32_t o = 0; o < S; ++o)
                            if (o != me) mbar_arrive_remote(mapa_u32(peer_ready_bar, slice_rank(o)));
                }
                bool cok = own_area || wait_bar_cluster(peer_ready_bar, 0, ctl, SITE_CLUSTER);
                if (named_bar_any(1, kEpiThreads, !cok)) break;
                const uint32_t row16 = (uint32_t)(q * 32 + lane) * 16u;
                if (e_swap_ab) {
                    // Same protocol; each lane holds one output column (its TMEM
                    // row) and 16 output rows per chunk.
                    for (int32_t h = 0; h < halves; ++h) {
#pragma unroll 1
                        for (int ci = 0; ci < 4; ++ci) {
                            const int32_t c = cg + 2 * ci;
                            if (c >= chunks) break;
                            const int32_t b = h * chunks + c, j = b / gsz, o = j % S;
                            if (o == me) continue;
                            const int32_t ob = (j / S) * gsz + (b - j * gsz);
                            const uint32_t slot = (uint32_t)(ob * (S - 1) + (me < o ? me : me - 1));
                            float v[16];
                            tmem_load_chunk<16>(tacc + (uint32_t)(h * e_bn + c * 16), v);
                            const uint32_t dst = mapa_u32(rbase + slot * kRedBlockBytes + row16, slice_rank(o));
                            const uint32_t rbar = mapa_u32(recv_bar, slice_rank(o));
#pragma unroll
                            for (int j4 = 0; j4 < 4; ++j4)
                                st_async_v4(dst + (uint32_t)j4 * 2048u, v[4 * j4], v[4 * j4 + 1], v[4 * j4 + 2],
                                            v[4 * j4 + 3], rbar);
                        }
                    }
                    cok = wait_bar_cluster(recv_bar, 0, ctl, SITE_CLUSTER);
                    if (named_bar_any(1, kEpiThreads, !cok)) break;
                    for (int32_t h = 0; h < halves; ++h) {
#pragma unroll 1
                        for (int ci = 0; ci < 4; ++ci) {
                            const int32_t c = cg + 2 * ci;
                            if (c >= chunks) break;
                            const int32_t b = h * chunks + c, j = b / gsz;
                            if (j % S != me) continue;
                            const int32_t ob = (j / S) * gsz + (b - j * gsz);
                            float v[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) v[i] = 0.0f;
#pragma unroll 1
                            for (int32_t s = 0; s < S; ++s) {
                                if (s == me) {
                                    float t[16];
                                    tmem_load_chunk<16>(tacc + (uint32_t)(h * e_bn + c * 16), t);
#pragma unroll
                                    for (int i = 0; i < 16; ++i) v[i] += t[i];
                                } else {
                                    const uint32_t slot = (uint32_t)(ob * (S - 1) + (s < me ? s : s - 1));
                                    const uint32_t src = rbase + slot * kRedBlockBytes + row16;
#pragma unroll
                                    for (int j4 = 0; j4 < 4; ++j4) {
                                        const float4 t = ld_shared_v4(src + (uint32_t)j4 * 2048u);
                                        v[4 * j4] += t.x;
                                        v[4 * j4 + 1] += t.y;
                                        v[4 * j4 + 2] += t.z;
                                        v[4 * j4 + 3] += t.w;
                                    }
                                }
                            }
                            bias_act_cols(v, h == 0 ? brow[0] : brow[1], e_epi, e_alpha);
                            const int32_t xn = r0 + h * 128 + q * 32;  // output column block (user N)
                            const int32_t ym = c0 + c * 16;            // output row block (user M)
                            if (e_res) add_residual_cols<ODT>(v, e_resid, e_rows, ym, xn + lane, e_cols, e_rows);
                            store_cols_chunk<ODT>(&tmC, ring, v, lane, xn, ym, xn < e_rows && ym < e_cols);
                        }
                    }
                    release_acc(acc);
                    if (++acc == e_n_acc) {
                        acc = 0;
                        acc_phase ^= 1u;
                    }
                    continue;
                }
                for (int32_t h = 0; h < halves; ++h) {
#pragma unroll 1
                    for (int ci = 0; ci < 4; ++ci) {
                        const int32_t c = cg + 2 * ci;
                        if (c >= chunks) break;
                        const int32_t b = h * chunks + c, j = b / gsz, o = j % S;
                        if (o == me) continue;
                        const int32_t ob = (j / S) * gsz + (b - j * gsz);
                        const uint32_t slot = (uint32_t)(ob * (S - 1) + (me < o ? me : me - 1));
                        float v[32];
                        tmem_load_chunk<32>(tacc + (uint32_t)(h * e_bn + c * 32), v);
                        const uint32_t dst = mapa_u32(rbase + slot * kRedBlockBytes + row16, slice_rank(o));
                        const uint32_t rbar = mapa_u32(recv_bar, slice_rank(o));
#pragma unroll
                        for (int j4 = 0; j4 < 8; ++j4)
                            st_async_v4(dst + (uint32_t)j4 * 2048u, v[4 * j4], v[4 * j4 + 1], v[4 * j4 + 2],
                                        v[4 * j4 + 3], rbar);
                    }
                }
                cok = wait_bar_cluster(recv_bar, 0, ctl, SITE_CLUSTER);
                if (named_bar_any(1, kEpiThreads, !cok)) break;
                for (int32_t h = 0; h < halves; ++h) {
#pragma unroll 1
                    for (int ci = 0; ci < 4; ++ci) {
                        const int32_t c = cg + 2 * ci;
                        if (c >= chunks) break;
                        const int32_t b = h * chunks + c, j = b / gsz;
                        if (j % S != me) continue;
                        const int32_t ob = (j / S) * gsz + (b - j * gsz);
                        float v[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = 0.0f;
#pragma unroll 1
                        for (int32_t s = 0; s < S; ++s) {
                            if (s == me) {
                                // own partial, straight from TMEM, 16 columns at a time
#pragma unroll
                                for (int hh = 0; hh < 2; ++hh) {
                                    float t[16];
                                    tmem_load_chunk<16>(tacc + (uint32_t)(h * e_bn + c * 32 + hh * 16), t);
#pragma unroll
                                    for (int i = 0; i < 16; ++i) v[hh * 16 + i] += t[i];
                                }
                            } else {
                                const uint32_t slot = (uint32_t)(ob * (S - 1) + (s < me ? s : s - 1));
                                const uint32_t src = rbase + slot * kRedBlockBytes + row16;
#pragma unroll
                                for (int j4 = 0; j4 < 8; ++j4) {
                                    const float4 t = ld_shared_v4(src + (uint32_t)j4 * 2048u);
                                    v[4 * j4] += t.x;
                                    v[4 * j4 + 1] += t.y;
                                    v[4 * j4 + 2] += t.z;
                                    v[4 * j4 + 3] += t.w;
                                }
                            }
                        }
                        bias_act_rows(v, bcol[ci], e_epi, e_alpha);
                        const int32_t n = c0 + c * 32, y = r0 + h * 128 + q * 32;
                        if (e_res) add_residual_rows<ODT>(v, e_resid, e_cols, y + lane, n, e_rows, e_cols);
                        store_rows_chunk<ODT>(&tmC, ring, v, lane, n, y, n < e_cols && y < e_rows);
                    }
                }
                release_acc(acc);
                if (++acc == e_n_acc) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
                continue;
            }
            if (e_coop && !e_swap_ab) {
                // One-wave split-K (one unit per CTA), finalised share by share.
                // The tile is cut into 32-row x 32-column blocks; block (row group
                // rg, chunk c) belongs to share (c/2 + max(1, chunks/2)*rg) mod S,
                // which gives every epilogue warp an even part of every share.
                // Share j has its own arrival count (S per launch; the counts only
                // grow).  Slice s writes the blocks of every other share to the
                // workspace ([slice][block][4-column group][32 rows][4], 4 KB per
                // block) and arrives on those shares.  It then waits, for a bounded
                // time, for the other S - 1 slices to arrive on its own share: if
                // they do, it adds the S partials of its blocks in slice order
                // (its own straight from TMEM) and runs the epilogue.  If they do
                // not (a slice that is not resident, its SM held by another
                // kernel), it writes its own blocks too and arrives; the slice
                // whose arrival completes a share's count finalises that share
                // from the workspace.  Nothing ever waits for a slice that may not
                // run, and every route sums in slice order, so all give the same bits.
                const int32_t S = e_split_k, me = w.split;
                const int32_t half_chunks = chunks >= 2 ? chunks / 2 : 1;
                const int32_t nblocks = (cta_rows / 32) * chunks;
                // Per-warp fetch region in the ring: R blocks of 4 KB (R >= 1).
                const int32_t fetch_r = max(1, min(S, (int32_t)(p.off_staging / (kEpiWarps * 4096u))));
                const uint32_t fetch_base = base + (uint32_t)ew * (uint32_t)fetch_r * 4096u;
                float4 *const xws = reinterpret_cast<float4 *>(e_workspace + (size_t)xtile * S * (size_t)tile_elems);
                uint64_t *const counts = e_epochs + (size_t)xtile * S;
                // This slice's partial of the blocks of share j (j < 0: of every
                // share but its own) -> workspace.
                auto write_blocks = [&](int32_t j) {
                    for (int32_t h = 0; h < halves; ++h) {
                        const int32_t rg = h * 4 + q;
#pragma unroll 1
                        for (int ci = 0; ci < 4; ++ci) {
                            const int32_t c = cg + 2 * ci;
                            if (c >= chunks) break;
                            const int32_t owner = (c / 2 + half_chunks * rg) % S;
                            if (j < 0 ? owner == me : owner != j) continue;
                            float v[32];
                            if (nk > 0) tmem_load_chunk<32>(tacc + (uint32_t)(h * e_bn + c * 32), v);
                            else {
#pragma unroll
                                for (int t = 0; t < 32; ++t) v[t] = 0.0f;
                            }
                            float4 *dst = xws + (size_t)(me * nblocks + rg * chunks + c) * 256 + lane;
#pragma unroll
                            for (int j4 = 0; j4 < 8; ++j4)
                                dst[j4 * 32] = make_float4(v[4 * j4], v[4 * j4 + 1], v[4 * j4 + 2], v[4 * j4 + 3]);
                        }
                    }
                };
                // Sum of the S partials of share j's blocks in slice order, then
                // the epilogue.  This slice's partial comes from TMEM when
                // `own_tmem` (the accumulator is still held), else from the
                // workspace like the others'.  The other blocks are fetched R at
                // a time with cp.async into this warp's region of the (idle)
                // pipeline ring, each thread reading back only its own pieces.
                auto finalise_share = [&](int32_t j, bool own_tmem) {
                    for (int32_t h = 0; h < halves; ++h) {
                        const int32_t rg = h * 4 + q;
#pragma unroll 1
                        for (int ci = 0; ci < 4; ++ci) {
                            const int32_t c = cg + 2 * ci;
                            if (c >= chunks) break;
                            if ((c / 2 + half_chunks * rg) % S != j) continue;
                            const float4 *src = xws + (size_t)(rg * chunks + c) * 256 + lane;
                            float v[32];
#pragma unroll
                            for (int t = 0; t < 32; ++t) v[t] = 0.0f;
#pragma unroll 1
                            for (int32_t s = 0; s < S;) {
                                int32_t s_end = s, got = 0;
                                while (s_end < S && (got < fetch_r || (s_end == me && own_tmem))) {
                                    if (!(s_end == me && own_tmem)) {
                                        const uint32_t dst = fetch_base + (uint32_t)got * 4096u + (uint32_t)lane * 16u;
                                        const float4 *g = src + (size_t)s_end * nblocks * 256;
#pragma unroll
                                        for (int j4 = 0; j4 < 8; ++j4)
                                            cp_async_16(dst + (uint32_t)j4 * 512u, g + j4 * 32);
                                        ++got;
                                    }
                                    ++s_end;
                                }
                                cp_async_commit_wait_all();
                                int32_t slot = 0;
                                for (; s < s_end; ++s) {
                                    if (s == me && own_tmem) {
                                        if (nk > 0) {
#pragma unroll
                                            for (int hh = 0; hh < 2; ++hh) {
                                                float o[16];
                                                tmem_load_chunk<16>(tacc + (uint32_t)(h * e_bn + c * 32 + hh * 16),
                                                                    o);
#pragma unroll
                                                for (int t = 0; t < 16; ++t) v[hh * 16 + t] += o[t];
                                            }
                                        }
                                    } else {
                                        const uint32_t from =
                                            fetch_base + (uint32_t)slot * 4096u + (uint32_t)lane * 16u;
#pragma unroll
                                        for (int j4 = 0; j4 < 8; ++j4) {
                                            const float4 t = ld_shared_v4(from + (uint32_t)j4 * 512u);
                                            v[4 * j4] += t.x;
                                            v[4 * j4 + 1] += t.y;
                                            v[4 * j4 + 2] += t.z;
                                            v[4 * j4 + 3] += t.w;
                                        }
                                        ++slot;
                                    }
                                }
                            }
                            bias_act_rows(v, bcol[ci], e_epi, e_alpha);
                            const int32_t n = c0 + c * 32, y = r0 + rg * 32;
                            if (e_res) add_residual_rows<ODT>(v, e_resid, e_cols, y + lane, n, e_rows, e_cols);
                            store_rows_chunk<ODT>(&tmC, ring, v, lane, n, y, n < e_cols && y < e_rows);
                        }
                    }
                };
                write_blocks(-1);
                named_bar_sync(1, kEpiThreads);
                // One warp arrives on the other shares (lane i on share me+1+i),
                // learning which of them it completes, and waits on its own.
                if (ew == 0) {
                    bool last = false;
                    if (lane < S - 1) {
                        const int32_t j = (me + 1 + lane) % S;
                        last = atom_acq_rel_gpu_add_u64(counts + j, 1) % (uint64_t)S == (uint64_t)(S - 1);
                    }
                    const uint32_t foreign = __ballot_sync(0xFFFFFFFFu, last);
                    uint32_t own = 0;
                    if (lane == 0) {
                        own = poll_share(counts + me, (uint32_t)S, ctl, p.share_poll_cycles) ? 1u : 0u;
                        if (own) atomicAdd(reinterpret_cast<unsigned long long *>(counts + me), 1ull);
                    }
                    own = __shfl_sync(0xFFFFFFFFu, own, 0);
                    // bit i: share me+1+i to finalise; bit 31: own share ready
                    if (lane == 0) *last_flag = (int32_t)(foreign | (own << 31));
                }
                named_bar_sync(1, kEpiThreads);
                const uint32_t flags = (uint32_t)*last_flag;
                named_bar_sync(1, kEpiThreads);   // the flag is rewritten below
                if (flags >> 31) {
                    finalise_share(me, true);
                } else {
                    // Hand the share over: publish this slice's own partial too.
                    write_blocks(me);
                    named_bar_sync(1, kEpiThreads);
                    if (ew == 0 && lane == 0)
                        *last_flag = atom_acq_rel_gpu_add_u64(counts + me, 1) % (uint64_t)S == (uint64_t)(S - 1);
                    named_bar_sync(1, kEpiThreads);
                    const bool mine = *last_flag != 0;
                    named_bar_sync(1, kEpiThreads);
                    if (mine) finalise_share(me, true);
                }
                release_acc(acc);
                if (++acc == e_n_acc) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
                for (int32_t i = 0; i < S - 1; ++i)
                    if ((flags >> i) & 1u) finalise_share((me + 1 + i) % S, false);
                continue;
            }
            float *ws = nullptr;
            if (e_split_k > 1) ws = e_workspace + ((size_t)xtile * e_split_k + w.split) * (size_t)tile_elems;

            for (int32_t h = 0; h < halves; ++h) {
                const int32_t r = h * 128 + q * 32 + lane;
                if (e_epi >= 7) {
                    // Gated epilogue (unswapped, one slice, the planner's rule):
                    // accumulator chunks 2p (gate) and 2p + 1 (up) of the fused
                    // tile give output chunk p, columns c0/2 + 32p of C [M, N/2].
#pragma unroll 1
                    for (int pi = 0; pi < 2; ++pi) {
                        const int32_t pp = cg + 2 * pi;
                        if (2 * pp >= chunks) break;
                        float g[32], u[32];
                        if (nk > 0) {
                            tmem_load_chunk<32>(tacc + (uint32_t)(h * e_bn + 2 * pp * 32), g);
                            tmem_load_chunk<32>(tacc + (uint32_t)(h * e_bn + 2 * pp * 32 + 32), u);
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j) g[j] = u[j] = 0.0f;
                        }
                        const float gb = load_bias1<ODT>(e_bias, c0 + 64 * pp + lane, e_cols);
                        const float ub = load_bias1<ODT>(e_bias, c0 + 64 * pp + 32 + lane, e_cols);
                        glu_rows(g, u, gb, ub, e_epi, e_alpha);
                        const int32_t n = (c0 >> 1) + pp * 32, y = r0 + h * 128 + q * 32;
                        store_rows_chunk<ODT>(&tmC, ring, g, lane, n, y, n < (e_cols >> 1) && y < e_rows);
                    }
                } else if (!e_swap_ab) {
#pragma unroll
                    for (int ci = 0; ci < 4; ++ci) {
                        const int32_t c = cg + 2 * ci;
                        if (c >= chunks) break;
                        float v[32];
                        if (nk > 0) tmem_load_chunk<32>(tacc + (uint32_t)(h * e_bn + c * 32), v);
                        else {
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[j] = 0.0f;
                        }
                        if (e_split_k > 1) {
                            float4 *dst = reinterpret_cast<float4 *>(ws);
#pragma unroll
                            for (int j4 = 0; j4 < 8; ++j4)
                                dst[(size_t)(c * 8 + j4) * cta_rows + r] =
                                    make_float4(v[4 * j4], v[4 * j4 + 1], v[4 * j4 + 2], v[4 * j4 + 3]);
                        } else {
                            bias_act_rows(v, bcol[ci], e_epi, e_alpha);
                            const int32_t n = c0 + c * 32, y = r0 + h * 128 + q * 32;
                            if (e_res) add_residual_rows<ODT>(v, e_resid, e_cols, y + lane, n, e_rows, e_cols);
                            store_rows_chunk<ODT>(&tmC, ring, v, lane, n, y, n < e_cols && y < e_rows);
                        }
                    }
                } else {
                    for (int32_t c = cg; c < chunks; c += 2) {
                        float v[16];
                        if (nk > 0) tmem_load_chunk<16>(tacc + (uint32_t)(h * e_bn + c * 16), v);
                        else {
#pragma unroll
                            for (int j = 0; j < 16; ++j) v[j] = 0.0f;
                        }
                        if (e_split_k > 1) {
                            float4 *dst = reinterpret_cast<float4 *>(ws);
#pragma unroll
                            for (int j4 = 0; j4 < 4; ++j4)
                                dst[(size_t)(c * 4 + j4) * cta_rows + r] =
                                    make_float4(v[4 * j4], v[4 * j4 + 1], v[4 * j4 + 2], v[4 * j4 + 3]);
                        } else {
                            bias_act_cols(v, h == 0 ? brow[0] : brow[1], e_epi, e_alpha);
                            const int32_t xn = r0 + h * 128 + q * 32;  // output column block (user N)
                            const int32_t ym = c0 + c * 16;            // output row block (user M)
                            if (e_res) add_residual_cols<ODT>(v, e_resid, e_rows, ym, xn + lane, e_cols, e_rows);
                            store_cols_chunk<ODT>(&tmC, ring, v, lane, xn, ym, xn < e_rows && ym < e_cols);
                        }
                    }
                }
            }
            // The accumulator may be overwritten by the next unit's MMAs.
            release_acc(acc);
            if (++acc == e_n_acc) {
                acc = 0;
                acc_phase ^= 1u;
            }

            if (e_split_k > 1) {
                // Split-K fix-up; every slice has written its whole partial.  One
                // wave (swapped tiles here; unswapped ones take the path above):
                // block b belongs to share b mod S, share j has its own arrival
                // count, and each slice arrives on the other shares, then waits a
                // bounded time on its own; the slice whose arrival completes a
                // share's count finalises it, and an owner whose peers all
                // arrived in time finalises its own.  Otherwise the last slice to
                // arrive on the tile's counter finalises the whole tile and resets
                // the count.  Either way the partials are summed in slice order.
                // The releases (after the CTA barrier that orders every epilogue
                // thread's partial stores before them) publish this CTA's
                // partial; the acquires, passed on by the next CTA barrier, make
                // the other slices' partials visible to every epilogue thread.
                named_bar_sync(1, kEpiThreads);
                if (ew == 0) {
                    uint32_t shares = 0;   // bit j: finalise share j (last arriver: bit 0, the tile)
                    if (e_coop) {
                        const int32_t S = e_split_k, me = w.split;
                        uint64_t *const counts = e_epochs + (size_t)xtile * S;
                        bool last = false;
                        if (lane < S - 1)
                            last = atom_acq_rel_gpu_add_u64(counts + (me + 1 + lane) % S, 1) % (uint64_t)S ==
                                   (uint64_t)(S - 1);
                        const uint32_t foreign = __ballot_sync(0xFFFFFFFFu, last);
                        uint32_t own = 0;
                        if (lane == 0) {
                            if (poll_share(counts + me, (uint32_t)S, ctl, p.share_poll_cycles)) {
                                atomicAdd(reinterpret_cast<unsigned long long *>(counts + me), 1ull);
                                own = 1;
                            } else {
                                own = atom_acq_rel_gpu_add_u64(counts + me, 1) % (uint64_t)S == (uint64_t)(S - 1);
                            }
                        }
                        own = __shfl_sync(0xFFFFFFFFu, own, 0);
                        for (int32_t i = 0; i < S - 1; ++i)
                            if ((foreign >> i) & 1u) shares |= 1u << ((me + 1 + i) % S);
                        if (own) shares |= 1u << me;
                    } else if (lane == 0) {
                        const int32_t old = atom_acq_rel_gpu_add(e_counters + xtile, 1);
                        if (old == e_split_k - 1) {
                            shares = 1;
                            atomicExch(e_counters + xtile, 0);
                        }
                    }
                    if (lane == 0) *last_flag = (int32_t)shares;
                }
                named_bar_sync(1, kEpiThreads);
                const uint32_t shares = (uint32_t)*last_flag;
                named_bar_sync(1, kEpiThreads);   // the flag is rewritten by the next unit
                const float4 *tile_ws =
                    reinterpret_cast<const float4 *>(e_workspace + (size_t)xtile * e_split_k * (size_t)tile_elems);
                const size_t slice4 = (size_t)tile_elems / 4;
                const int32_t rgroups = cta_rows / 32;
                const int32_t nblocks = rgroups * chunks;
                const int32_t n_shares = e_coop ? e_split_k : 1;
#pragma unroll 1
                for (int32_t jsh = 0; jsh < n_shares; ++jsh) {
                    if (!((shares >> jsh) & 1u)) continue;
                    const int32_t first_b = jsh, stride = n_shares;
                    for (int32_t b = first_b + stride * ew; b < nblocks; b += stride * kEpiWarps) {
                        const int32_t rg = b % rgroups, c = b / rgroups;
                        const int32_t r = rg * 32 + lane;
                        if (!e_swap_ab) {
                            float v[32];
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[j] = 0.0f;
                            const float4 *src = tile_ws + (size_t)(c * 8) * cta_rows + r;
                            const float lb = e_epi != 0 ? load_bias1<ODT>(e_bias, c0 + c * 32 + lane, e_cols) : 0.0f;
                            for (int32_t s = 0; s < e_split_k; ++s) {
                                float4 t[8];
#pragma unroll
                                for (int j4 = 0; j4 < 8; ++j4) t[j4] = __ldcg(src + s * slice4 + (size_t)j4 * cta_rows);
#pragma unroll
                                for (int j4 = 0; j4 < 8; ++j4) {
                                    v[4 * j4] += t[j4].x;
                                    v[4 * j4 + 1] += t[j4].y;
                                    v[4 * j4 + 2] += t[j4].z;
                                    v[4 * j4 + 3] += t[j4].w;
                                }
                            }
                            bias_act_rows(v, lb, e_epi, e_alpha);
                            const int32_t n = c0 + c * 32, y = r0 + rg * 32;
                            if (e_res) add_residual_rows<ODT>(v, e_resid, e_cols, y + lane, n, e_rows, e_cols);
                            store_rows_chunk<ODT>(&tmC, ring, v, lane, n, y, n < e_cols && y < e_rows);
                        } else {
                            float v[16];
#pragma unroll
                            for (int j = 0; j < 16; ++j) v[j] = 0.0f;
                            const float4 *src = tile_ws + (size_t)(c * 4) * cta_rows + r;
                            const float rb = e_epi != 0 ? load_bias1<ODT>(e_bias, r0 + r, e_rows) : 0.0f;
                            for (int32_t s = 0; s < e_split_k; s += 4) {
                                float4 t[4][4];
#pragma unroll
                                for (int i = 0; i < 4; ++i)
                                    if (s + i < e_split_k) {
#pragma unroll
                                        for (int j4 = 0; j4 < 4; ++j4)
                                            t[i][j4] = __ldcg(src + (s + i) * slice4 + (size_t)j4 * cta_rows);
                                    }
#pragma unroll
                                for (int i = 0; i < 4; ++i)
                                    if (s + i < e_split_k) {
#pragma unroll
                                        for (int j4 = 0; j4 < 4; ++j4) {
                                            v[4 * j4] += t[i][j4].x;
                                            v[4 * j4 + 1] += t[i][j4].y;
                                            v[4 * j4 + 2] += t[i][j4].z;
                                            v[4 * j4 + 3] += t[i][j4].w;
                                        }
                                    }
                            }
                            bias_act_cols(v, rb, e_epi, e_alpha);
                            const int32_t xn = r0 + rg * 32, ym = c0 + c * 16;
                            if (e_res) add_residual_cols<ODT>(v, e_resid, e_rows, ym, xn + lane, e_cols, e_rows);
                            store_cols_chunk<ODT>(&tmC, ring, v, lane, xn, ym, xn < e_rows && ym < e_cols);
                        }
                    }
                }
            }
        }
        if (lane == 0) bulk_wait_all();
    }

    __syncthreads();
    // A CTA pair touches each other's barriers, shared memory and TMEM until
    // both are done: neither leaves (or frees TMEM) before the other.
    if (pair) cluster_sync_all();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc<CG>(tmem_base, p.tmem_cols);
    }
}

// Counter-based 32-bit hash of element i (a finaliser of the splitmix family).
__device__ __forceinline__ uint32_t hash_u32(uint32_t x)
{
    x ^= x >> 16;
    x *= 0x7FEB352Du;
    x ^= x >> 15;
    x *= 0x846CA68Bu;
    x ^= x >> 16;
    return x;
}

// Fills a buffer with counter-based pseudo-random values: dist 0 uniform in
// [-scale, scale], dist 1 normal with standard deviation `scale` (Box-Muller
// on two hashed uniforms).  Tuning inputs only, never user data.
__global__ void fill_random_kernel(void *dst, int64_t n, int dt, float scale, uint32_t seed, int dist)
{
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const uint32_t x = hash_u32((uint32_t)i * 0x9E3779B9u ^ seed);
        float f;
        if (dist == 0) {
            f = ((float)(x >> 8) * (1.0f / 16777216.0f) * 2.0f - 1.0f) * scale;
        } else {
            const uint32_t y = hash_u32(x ^ 0x68E31DA4u ^ (uint32_t)(i >> 32));
            const float u1 = ((float)(x >> 8) + 1.0f) * (1.0f / 16777216.0f);   // (0, 1]
            const float u2 = (float)(y >> 8) * (1.0f / 16777216.0f);
            f = sqrtf(-2.0f * logf(u1)) * cospif(2.0f * u2) * scale;
        }
        if (dt == 0) reinterpret_cast<__nv_bfloat16 *>(dst)[i] = __float2bfloat16_rn(f);
        else if (dt == 2 || dt == 3) reinterpret_cast<__nv_fp8_storage_t *>(dst)[i] = __nv_cvt_float_to_fp8(f, __NV_SATFINITE, __NV_E4M3);
        else reinterpret_cast<float *>(dst)[i] = f;
    }
}

// Row-major [rows, cols] -> row-major [cols, rows] through 32x32 shared-memory
// tiles, so that both the reads and the writes are coalesced.  Used to give the
// tensor cores a K-major copy of B when B must not be read MN-major.
// Byte matrix transpose (an FP8 operand's K-major copy), rows and cols
// multiples of 4: each thread reads a 4 x 4 block of bytes as four 32-bit words
// (one per row; a warp covers 4 rows x 32 columns), transposes it in registers
// with byte permutes, and the resulting words (4 consecutive rows of one
// column each) are transposed as 32-bit elements through shared memory, so
// that both the reads and the writes are whole 32-bit words along rows.  A
// block moves 128 rows x 32 columns per step.
__global__ void __launch_bounds__(256) transpose_bytes_kernel(const uint8_t *__restrict__ src,
                                                              uint8_t *__restrict__ dst, int64_t rows, int64_t cols)
{
    __shared__ uint32_t tile[32][33];    // [row quad][column]
    const int t = threadIdx.x;
    const int g = t & 7, q = t >> 3;     // column group of 4, row quad
    const int64_t c0 = (int64_t)blockIdx.x * 32;
    const uint32_t *s32 = reinterpret_cast<const uint32_t *>(src);
    uint32_t *d32 = reinterpret_cast<uint32_t *>(dst);
    const int64_t cw = cols / 4, rw = rows / 4;   // row lengths in words
    for (int64_t r0 = (int64_t)blockIdx.y * 128; r0 < rows; r0 += (int64_t)gridDim.y * 128) {
        const int64_t r = r0 + 4 * q, c = c0 + 4 * g;
        uint32_t w0 = 0, w1 = 0, w2 = 0, w3 = 0;
        if (r < rows && c < cols) {
            const int64_t i = r * cw + c / 4;
            w0 = __ldg(s32 + i);
            w1 = __ldg(s32 + i + cw);
            w2 = __ldg(s32 + i + 2 * cw);
            w3 = __ldg(s32 + i + 3 * cw);
        }
        // Word j of the result holds column c + j of rows r .. r + 3 (byte k = row r + k).
        const uint32_t lo01 = __byte_perm(w0, w1, 0x5140), hi01 = __byte_perm(w0, w1, 0x7362);
        const uint32_t lo23 = __byte_perm(w2, w3, 0x5140), hi23 = __byte_perm(w2, w3, 0x7362);
        tile[q][4 * g + 0] = __byte_perm(lo01, lo23, 0x5410);
        tile[q][4 * g + 1] = __byte_perm(lo01, lo23, 0x7632);
        tile[q][4 * g + 2] = __byte_perm(hi01, hi23, 0x5410);
        tile[q][4 * g + 3] = __byte_perm(hi01, hi23, 0x7632);
        __syncthreads();
        // Column c0 + n of the source is row c0 + n of the destination; its
        // words r0/4 + 0 .. 31 are tile[0 .. 31][n].
        const int lq = t & 31;
        for (int n = t >> 5; n < 32; n += 8) {
            const int64_t dr = c0 + n, dq = r0 / 4 + lq;
            if (dr < cols && dq < rw) d32[dr * rw + dq] = tile[lq][n];
        }
        __syncthreads();
    }
}

template <typename T>
__global__ void transpose_kernel(const T *__restrict__ src, T *__restrict__ dst, int64_t rows, int64_t cols)
{
    __shared__ T tile[32][33];
    const int64_t c0 = (int64_t)blockIdx.x * 32;
    for (int64_t r0 = (int64_t)blockIdx.y * 32; r0 < rows; r0 += (int64_t)gridDim.y * 32) {
        for (int i = threadIdx.y; i < 32; i += 8) {
            const int64_t r = r0 + i, c = c0 + threadIdx.x;
            if (r < rows && c < cols) tile[i][threadIdx.x] = src[r * cols + c];
        }
        __syncthreads();
        for (int i = threadIdx.y; i < 32; i += 8) {
            const int64_t c = c0 + i, r = r0 + threadIdx.x;
            if (c < cols && r < rows) dst[c * rows + r] = tile[threadIdx.x][i];
        }
        __syncthreads();
    }
}

}  // namespace

// ---------------------------------------------------------------------------
// Host-side launch helpers
// ---------------------------------------------------------------------------

// Kernel instances: (dtype, A MN-major, B MN-major, CTA group).  bf16 reads B
// MN-major in place (unswapped: B is MMA-B; swapped: B is MMA-A); fp32 reads
// both operands K-major from a transposed copy of B.  A kernel may not mix
// single-CTA and CTA-pair tcgen05 instructions, so pairs are instances of their
// own (unswapped only).
template <int DT, bool AM, bool BM, int CG>
static const void *kernel_fn()
{
    return reinterpret_cast<const void *>(gemm_tcgen05_kernel<DT, AM, BM, CG>);
}

static const void *select_kernel(int dt, int a_mn, int b_mn, int cg)
{
    if (dt == 3) {   // block-scaled FP8: B in place (unswapped: MMA-B; swapped: MMA-A) or K-major; pairs unswapped
        if (cg == 2) {
            if (a_mn) return nullptr;
            return b_mn ? kernel_fn<3, false, true, 2>() : kernel_fn<3, false, false, 2>();
        }
        if (!a_mn && b_mn) return kernel_fn<3, false, true, 1>();
        if (a_mn && !b_mn) return kernel_fn<3, true, false, 1>();
        if (!a_mn && !b_mn) return kernel_fn<3, false, false, 1>();
        return nullptr;
    }
    if (cg == 2) {
        if (a_mn) return nullptr;
        if (dt == 0) return b_mn ? kernel_fn<0, false, true, 2>() : kernel_fn<0, false, false, 2>();
        if (dt == 2) return b_mn ? kernel_fn<2, false, true, 2>() : kernel_fn<2, false, false, 2>();
        return b_mn ? nullptr : kernel_fn<1, false, false, 2>();
    }
    if (dt == 2) {   // FP8, like bf16: B MN-major in place (unswapped: MMA-B; swapped: MMA-A), or K-major copy
        if (!a_mn && b_mn) return kernel_fn<2, false, true, 1>();
        if (a_mn && !b_mn) return kernel_fn<2, true, false, 1>();
        if (!a_mn && !b_mn) return kernel_fn<2, false, false, 1>();
        return nullptr;
    }
    if (dt == 0) {
        if (!a_mn && b_mn) return kernel_fn<0, false, true, 1>();
        if (a_mn && !b_mn) return kernel_fn<0, true, false, 1>();
        if (!a_mn && !b_mn) return kernel_fn<0, false, false, 1>();
        return nullptr;
    }
    if (!a_mn && !b_mn) return kernel_fn<1, false, false, 1>();
    return nullptr;
}

// Every instance of a dtype: (A MN-major, B MN-major, CTA group).
static const int kInstances[5][3] = {{0, 1, 1}, {1, 0, 1}, {0, 0, 1}, {0, 1, 2}, {0, 0, 2}};

cudaError_t kernel_attributes(int dt, int *num_regs, int *max_threads)
{
    int regs = 0, thr = 1 << 30;
    for (const auto &c : kInstances) {
        const void *f = select_kernel(dt, c[0], c[1], c[2]);
        if (!f) continue;
        cudaFuncAttributes a;
        cudaError_t e = cudaFuncGetAttributes(&a, f);
        if (e != cudaSuccess) return e;
        if (a.numRegs > regs) regs = a.numRegs;
        if (a.maxThreadsPerBlock < thr) thr = a.maxThreadsPerBlock;
    }
    if (num_regs) *num_regs = regs;
    if (max_threads) *max_threads = thr;
    return cudaSuccess;
}

cudaError_t set_kernel_smem_limit(int dt, int bytes)
{
    for (const auto &c : kInstances) {
        const void *f = select_kernel(dt, c[0], c[1], c[2]);
        if (!f) continue;
        cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_gemm(int dt, const CUtensorMap &a, const CUtensorMap &b, const CUtensorMap &c,
                        const CUtensorMap *sa, const CUtensorMap *sb, const KernelParams &p, int grid, int smem_bytes,
                        cudaStream_t stream)
{
    const void *f = select_kernel(dt, p.a_mn_major, p.b_mn_major, p.pair ? 2 : 1);
    if (!f) return cudaErrorInvalidValue;
    // The MX scale maps are read only by block-scaled instances; others get zeros.
    static const CUtensorMap none{};
    void *args[] = {const_cast<CUtensorMap *>(&a),  const_cast<CUtensorMap *>(&b),
                    const_cast<CUtensorMap *>(&c),  const_cast<CUtensorMap *>(sa ? sa : &none),
                    const_cast<CUtensorMap *>(sb ? sb : &none), const_cast<KernelParams *>(&p)};
    // Every launch allows programmatic overlap with the previous kernel on the
    // stream (the kernel waits on griddepcontrol before touching memory).  No
    // CTA waits without bound for another (the split-K share owners' waits
    // fall back), so no launch needs to be cooperative.
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.cluster_k > 1) {
        // The K slices of a tile are one cluster (consecutive CTAs, or
        // consecutive pairs of a pair tile).
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)p.cluster_k * (p.pair ? 2u : 1u);
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    } else if (p.pair) {
        // A CTA pair is a cluster of two consecutive CTAs.
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 2;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    return cudaLaunchKernelExC(&cfg, f, args);
}

// Clusters of `cluster` CTAs of this kernel that fit on the device at once.
cudaError_t max_active_clusters(int dt, int a_mn, int b_mn, int cg, int cluster, int smem_bytes, int *out)
{
    *out = 0;
    const void *f = select_kernel(dt, a_mn, b_mn, cg);
    if (!f) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)cluster);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)smem_bytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(out, f, &cfg);
}

cudaError_t launch_transpose(const void *src, void *dst, int64_t rows, int64_t cols, int elt, cudaStream_t stream)
{
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    if (elt == 1 && rows % 4 == 0 && cols % 4 == 0 && ((uintptr_t)src & 3) == 0 && ((uintptr_t)dst & 3) == 0) {
        const int64_t gy = (rows + 127) / 128;
        const dim3 grid((unsigned)((cols + 31) / 32), (unsigned)(gy < 65535 ? gy : 65535));
        transpose_bytes_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint8_t *>(src),
                                                         static_cast<uint8_t *>(dst), rows, cols);
        return cudaGetLastError();
    }
    const int64_t gy = (rows + 31) / 32;
    const dim3 grid((unsigned)((cols + 31) / 32), (unsigned)(gy < 65535 ? gy : 65535));
    const dim3 block(32, 8);
    if (elt == 1)
        transpose_kernel<uint8_t><<<grid, block, 0, stream>>>(static_cast<const uint8_t *>(src),
                                                              static_cast<uint8_t *>(dst), rows, cols);
    else if (elt == 2)
        transpose_kernel<uint16_t><<<grid, block, 0, stream>>>(static_cast<const uint16_t *>(src),
                                                               static_cast<uint16_t *>(dst), rows, cols);
    else
        transpose_kernel<uint32_t><<<grid, block, 0, stream>>>(static_cast<const uint32_t *>(src),
                                                               static_cast<uint32_t *>(dst), rows, cols);
    return cudaGetLastError();
}

// MX scale packing: one thread per packed byte.  Packed byte o lies in atom
// o/512 = (row atom rt, K atom kt) of the KT K atoms per row atom; within the
// atom, byte (r%32)·16 + ((r%128)/32)·4 + j%4 holds the scale of row r, block
// j (32 elements of K).  Rows or blocks past the operand read as 0.
__global__ void mx_pack_kernel(const uint8_t *__restrict__ src, int64_t rows, int64_t kblocks, int64_t kt_atoms,
                               int64_t total, int b_side, uint8_t *__restrict__ dst)
{
    for (int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; o < total; o += (int64_t)gridDim.x * blockDim.x) {
        const int64_t atom = o >> 9;
        const int32_t within = (int32_t)(o & 511);
        const int64_t rt = atom / kt_atoms, kt = atom % kt_atoms;
        const int64_t r = rt * 128 + (within & 15) / 4 * 32 + within / 16;
        const int64_t j = kt * 4 + (within & 3);
        uint8_t v = 0;
        if (r < rows && j < kblocks) v = b_side ? src[j * rows + r] : src[r * kblocks + j];
        dst[o] = v;
    }
}

cudaError_t launch_mx_pack(const uint8_t *src, int64_t rows, int64_t K, int b_side, uint8_t *dst,
                           cudaStream_t stream)
{
    const int64_t rt = 2 * ((rows + 255) / 256), kt = 2 * ((K + 255) / 256);
    const int64_t total = rt * kt * 512;
    if (total <= 0) return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 8192) blocks = 8192;
    mx_pack_kernel<<<(unsigned)blocks, 256, 0, stream>>>(src, rows, (K + 31) / 32, kt, total, b_side, dst);
    return cudaGetLastError();
}

cudaError_t launch_fill_random(void *dst, int64_t n, int dt, float scale, uint32_t seed, int dist,
                               cudaStream_t stream)
{
    if (n <= 0) return cudaSuccess;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    fill_random_kernel<<<(unsigned)blocks, 256, 0, stream>>>(dst, n, dt, scale, seed, dist);
    return cudaGetLastError();
}

}  // namespace gemmgb
