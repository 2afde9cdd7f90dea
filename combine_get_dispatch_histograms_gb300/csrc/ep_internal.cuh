// ep_internal.cuh -- shared internals of libep_gb300: the context object,
// error plumbing, launch bookkeeping and the inline-PTX primitives (bulk
// async copies, mbarriers, acquire/release accesses) the kernels are built on.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <cstddef>

#include "ep.h"

namespace ep {

// ---- device status word bits ------------------------------------------------
enum : uint32_t {
    FLAG_INVALID_TOPK = 1u,  // topk_idx outside [-1, E)
    FLAG_CAPACITY = 2u,      // a region / buffer would overflow
    FLAG_TIMEOUT = 4u,       // a bounded wait ran out
    FLAG_BOUNDS = 8u,        // an internal index check failed (access skipped)
};

constexpr int kMaxRanks = 64;
constexpr int kMaxTopk = 32;
constexpr int kMaxLocalExperts = 1024;
constexpr int kMaxExperts = 4096;
constexpr int kTileTokens = 256;  // tokens per CTA of the layout / notify kernels
constexpr int kMaxDevicesTracked = 64;  // per-device launch attributes cached up to this index

// ---- host-side error plumbing -------------------------------------------------
ep_status set_error(ep_status st, const char* fmt, ...);
ep_status cuda_error(cudaError_t e, const char* what);
#define EP_CUDA(call)                                                   \
    do {                                                                \
        cudaError_t e__ = (call);                                       \
        if (e__ != cudaSuccess) return ::ep::cuda_error(e__, #call);    \
    } while (0)
#define EP_CHECK_LAUNCH(what)                                           \
    do {                                                                \
        cudaError_t e__ = cudaGetLastError();                           \
        if (e__ != cudaSuccess) return ::ep::cuda_error(e__, what);     \
    } while (0)
ep_status status_from_flags(uint32_t flags);
bool aligned16(const void* p);

// ---- geometry of the token tiles (layout / notify) -------------------------
// Channel c owns tokens [c*ct, min(T, (c+1)*ct)), ct = ceil(T / C); each channel
// is cut into ceil(ct / kTileTokens) tiles so that no tile straddles channels.
struct TileGeom {
    int T, C, ct, tiles_per_channel, tiles_per_src;
};
inline TileGeom make_tiles(int T, int C) {
    TileGeom g;
    g.T = T;
    g.C = C;
    g.ct = (T + C - 1) / C;
    if (g.ct < 1) g.ct = 1;
    g.tiles_per_channel = (g.ct + kTileTokens - 1) / kTileTokens;
    g.tiles_per_src = C * g.tiles_per_channel;
    return g;
}
__host__ __device__ inline void tile_range(const TileGeom& g, int tile, int* lo, int* hi) {
    int c = tile / g.tiles_per_channel, j = tile % g.tiles_per_channel;
    int a = c * g.ct + j * kTileTokens;
    int b = a + kTileTokens;
    int ce = (c + 1) * g.ct;
    if (b > ce) b = ce;
    if (b > g.T) b = g.T;
    if (a > g.T) a = g.T;
    *lo = a;
    *hi = b > a ? b : a;
}

}  // namespace ep

// ---- the context ----------------------------------------------------------------
struct ep_ctx {
    ep_config cfg;
    int device;
    int num_sms;
    int L, G;  // experts per rank, ranks per node
    ep::TileGeom tiles;
    // device workspace
    void* ws;
    size_t ws_bytes;
    int32_t* ws_layout_part;   // [R][tiles][E + R + N] partial counts of the layout kernel
    int32_t* ws_notify_part;   // [R][tiles][E + R + N] partial counts of the notify kernel
    int32_t* ws_ebase;         // [R][E]   first permuted row of (source, expert)
    int32_t* ws_sbase;         // [R][N]   first staging row of (source, node)
    uint32_t* ws_layout_done;  // [R]      per-source tile completion counters
    uint32_t* ws_notify_done;  // [1]
    uint32_t* status;          // [1]      device status word
    // pinned, device-mapped host block written by the notify kernel
    int32_t* host_block;       // [R + R*L + 8]: counts, totals, status, sequence word
    int32_t notify_epoch;      // sequence number of the last notify
    int32_t* host_block_dev;
    cudaEvent_t ev_counts;
    int64_t wait_timeout_ns;
    // copy-engine launch shape per route kind (ep::CopyKind), chosen at context
    // creation; environment variables override them for sweeps
    int copy_ctas_per_sm[4], copy_stage_bytes[4], copy_read_depth;
    bool copy_shape_forced[4];  // set from the environment: used as given
    // totals of the last notify (host copies), sizes of later launches
    int64_t last_total_recv, last_total_perm, last_total_stage;
    bool totals_known;  // false after a notify that did not wait for the counts
    int expert_alignment;  // rows of each permuted expert block are rounded up to this
    int last_launches;
};

namespace ep {

// route kinds of the copy engine, each with its own launch shape
enum CopyKind : int { COPY_PERMUTE = 0, COPY_SCATTER = 1, COPY_FUSED = 2, COPY_STAGE = 3 };

// ---- small device helpers -------------------------------------------------------
__device__ __forceinline__ void flag(uint32_t* status, uint32_t bits) { atomicOr(status, bits); }

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu(int* p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_gpu(int* p, int v) {
    asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// 16-byte streaming load through the non-coherent path, no L1 allocation
__device__ __forceinline__ int4 ld_nc_na_v4(const void* p) {
    int4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
// 16-byte store, no L1 allocation
__device__ __forceinline__ void st_na_v4(void* p, int4 v) {
    asm volatile("st.global.L1::no_allocate.v4.s32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// ---- mbarrier + bulk async copy (sm_90+ PTX, used here on sm_103a) -------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
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
// Bounded wait: returns false (and the caller flags a timeout) if the phase
// has not completed within `limit_ns`.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((int64_t)(globaltimer_ns() - t0) > limit_ns) return false;
    }
}
// global -> shared bulk copy completing on an mbarrier (bytes % 16 == 0, both 16-aligned)
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// shared -> global bulk copy tracked by the bulk-group mechanism
__device__ __forceinline__ void bulk_s2g(void* gmem_dst, const void* smem_src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gmem_dst),
                 "r"(smem_u32(smem_src)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---- row movers shared by the bf16 and fp8 entry points (ep_copy.cu) -------------
ep_status dispatch_rows(ep_ctx* c, const void* x, int64_t row_bytes, const int64_t* topk_idx, const float* topk_weights,
                        const ep_dispatch_handle* h, void* recv_x, int32_t* recv_src_rank, int32_t* recv_src_idx,
                        int32_t* recv_topk_idx, float* recv_topk_weights, int64_t recv_capacity_rows, void* stream);
ep_status permute_rows(ep_ctx* c, const ep_dispatch_handle* h, const void* recv_x, int64_t row_bytes,
                       const int32_t* recv_src_rank, const int32_t* recv_src_idx, const int32_t* recv_topk_idx,
                       int64_t num_recv_rows, void* permuted_x, int32_t* perm_src_row, int64_t perm_capacity_rows,
                       void* stream);
ep_status dispatch_permuted_rows(ep_ctx* c, const void* x, int64_t row_bytes, const int64_t* topk_idx,
                                 const float* topk_weights, const ep_dispatch_handle* h, void* permuted_x,
                                 int32_t* perm_src_token, float* perm_weight, int64_t perm_capacity_rows,
                                 void* stream);

// ---- launch helpers -------------------------------------------------------------
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace ep
