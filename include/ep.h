/*
 * ep.h -- C ABI of the GB300 (sm_103a) MoE expert-parallel dispatch / combine
 * library (libep_gb300.so).
 *
 * The operations follow three pages on DeepEP-style expert parallelism:
 *   [P1] "事件驱动 EP 内核的调度策略与零拷贝通信：从 DeepEP 看高性能并发架构设计"
 *        (sections 事件驱动调度的本质, 高吞吐量模式, 低延迟模式)
 *   [P2] "DeepEP 学习笔记：MoE 场景下的专家并行通信"
 *        (sections dispatch 前：全局布局与通知, dispatch 过程, combine 过程,
 *         三个方法概览, DeepEP v2 direct 模式, hybrid 模式)
 *   [P3] "DeepSeek DeepEP探索：低延迟分发（low latency dispatch）的架构设计与实现"
 *        (sections 2.2 显存管理的权衡策略, 4.2 接收端的自适应处理)
 *
 * Model.  R "ranks" are virtual partitions of ONE GPU's memory: every array
 * below is the concatenation over ranks of that rank's array, in one device
 * allocation.  E experts, L = E / R per rank, expert e lives on rank e / L.
 * K = top-k, T = tokens per source rank, H = hidden size (bf16 channels),
 * C = channels (token ranges) of the notify step, N = nodes (R % N == 0,
 * G = R / N ranks per node, rank r on node r / G).
 *
 * Conventions for every entry point:
 *   - Pointers named without "host_" are DEVICE pointers (cudaMalloc'd or
 *     torch tensors), caller-owned, row-major, contiguous.  Row arrays of bf16
 *     ([..][H]) and fp8 ([..][H]) must be 16-byte aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Every call is asynchronous on that stream, except
 *     ep_notify_dispatch and ep_layout_notify in their waiting forms (they
 *     wait for the receive counts, the one host synchronisation of the normal
 *     path) and the *_check calls.
 *   - bf16 values are passed as void* (2 bytes each); topk_idx is int64 with -1
 *     meaning "masked" (the entry is ignored everywhere); topk_weights fp32.
 *   - Return EP_OK or a negative ep_status; the message of the last failure on
 *     the calling thread is ep_last_error().  Arguments are validated on the
 *     host before any launch.  Errors found on the device (a topk_idx value
 *     outside [-1, E), a full low-latency region, a wait that ran out) are
 *     recorded in a device status word and reported by ep_ctx_check /
 *     ep_ll_check (the waiting notify reports them too, since it synchronises).
 */
#ifndef EP_GB300_H
#define EP_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ep_status {
    EP_OK = 0,
    EP_ERR_INVALID_ARG = -1,   /* bad pointer, size, alignment or configuration        */
    EP_ERR_INVALID_INPUT = -2, /* topk_idx holds a value outside [-1, E)                */
    EP_ERR_CAPACITY = -3,      /* a caller buffer or a low-latency region is too small  */
    EP_ERR_TIMEOUT = -4,       /* a bounded device wait ran out (count slot, copy)      */
    EP_ERR_CUDA = -5           /* a CUDA runtime call failed                            */
} ep_status;

/* Message of the last failure on the calling thread ("" if none). */
const char* ep_last_error(void);
/* Name of a status code, e.g. "EP_ERR_TIMEOUT". */
const char* ep_status_name(int status);
/* Library version string. */
const char* ep_version(void);

/* ------------------------------------------------------------------------ */
/* Context (the [P2] Buffer: owns workspace and the CPU-mapped counters)     */
/* ------------------------------------------------------------------------ */

typedef struct ep_config {
    int32_t num_ranks;    /* R, 1..64                                        */
    int32_t num_experts;  /* E, multiple of R, E / R <= 1024, E <= 4096       */
    int32_t num_topk;     /* K, 1..32                                        */
    int32_t num_tokens;   /* T, tokens per source rank, >= 0                  */
    int32_t hidden;       /* H, bf16 channels per token, multiple of 8        */
    int32_t num_channels; /* C, 1..1024: channel c owns tokens [c*ceil(T/C), ...) */
    int32_t num_nodes;    /* N, 1..R with R % N == 0 (1 = flat)              */
} ep_config;

typedef struct ep_ctx ep_ctx;

/* Creates a context on the current CUDA device.  Allocates the device
 * workspace (per-tile partial counts, a status word) and a pinned,
 * device-mapped host block for the receive counts ([P2] Buffer: "分配
 * workspace", "CPU-mapped counters").  Free with ep_ctx_destroy. */
ep_status ep_ctx_create(const ep_config* cfg, ep_ctx** out);
void ep_ctx_destroy(ep_ctx* ctx);

/* Synchronises `stream`, reads and clears the device status word.  Returns
 * EP_OK, EP_ERR_INVALID_INPUT, EP_ERR_CAPACITY or EP_ERR_TIMEOUT. */
ep_status ep_ctx_check(ep_ctx* ctx, void* stream);

/* Limit, in microseconds, of every bounded device wait of this context
 * (copy-pipeline barriers).  Default 2 000 000. */
ep_status ep_ctx_set_wait_timeout_us(ep_ctx* ctx, int64_t us);

/* Expert alignment of the permuted layout (default 1 = none; 1..65536, and
 * R*T*K + E*(alignment-1) below 2^31, else EP_ERR_INVALID_ARG).
 * The pages fix none; it serves a grouped GEMM that wants every expert's
 * block to start on a tile boundary.  From the next ep_notify_dispatch on,
 * each (rank d, local expert l) block of the permuted layout takes
 * num_recv_per_expert[d][l] rounded up to a multiple of `alignment` rows:
 * expert_offsets[d][l] (a multiple of the alignment), perm_rank_base and
 * the permuted totals include the padding; num_recv_per_expert stays the
 * pair count.  The pairs fill the first rows of their block in the usual
 * order; padding rows of permuted_x, perm_src_row, perm_src_token and
 * perm_weight are not written.  Combine reads only the pairs' rows. */
ep_status ep_ctx_set_expert_alignment(ep_ctx* ctx, int32_t alignment);
/* The context's current expert alignment (1 for a fresh context); 0 if ctx
 * is NULL. */
int32_t ep_ctx_expert_alignment(const ep_ctx* ctx);

/* Number of kernel launches the last call on this context made (for the
 * bench's launch count). */
int32_t ep_ctx_last_launches(const ep_ctx* ctx);

/* ------------------------------------------------------------------------ */
/* Layout: get_dispatch_layout  ([P2] dispatch 前：全局布局与通知)            */
/* ------------------------------------------------------------------------ */

/* From topk_idx [R][T][K] computes, per source rank s:
 *   num_tokens_per_expert [R][E] int32: valid (t,k) with topk_idx == e;
 *   num_tokens_per_rank   [R][R] int32: tokens t with is_token_in_rank[s][t][d];
 *   is_token_in_rank      [R][T][R] uint8: 1 iff some valid k has e / L == d
 *     (the top-k list flattened into a lookup table, one copy per rank);
 *   and, when both node pointers are non-NULL (hierarchical mode),
 *   num_tokens_per_node   [R][N] int32 and is_token_in_node [R][T][N] uint8.
 * Out-of-range topk_idx values are skipped and flagged (EP_ERR_INVALID_INPUT
 * at the next check). */
ep_status ep_get_dispatch_layout(ep_ctx* ctx, const int64_t* topk_idx,
                                 int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                                 uint8_t* is_token_in_rank, int32_t* num_tokens_per_node,
                                 uint8_t* is_token_in_node, void* stream);

/* Allocation-free layout.  The pages have no counterpart of this entry point;
 * it exists for callers that must not allocate device memory themselves: for
 * example a plug-in inside a serving runtime that owns every byte of HBM
 * through its own pool and hands out only the tensors it manages, or a
 * latency-critical path where cudaMalloc / cudaFree (which can synchronise
 * the whole device and can fail once the memory is reserved) are not allowed.
 * It computes exactly what ep_get_dispatch_layout computes, without a context:
 * its scratch (per-tile partial counts, per-source completion counters, a
 * status word) is a fixed array in the library's device memory of
 * EP_LAYOUT_NOALLOC_SCRATCH_BYTES, held by every GPU that loads the library
 * until the process exits.  It calls no allocating routine.
 *   - Sizes: num_ranks 1..64, num_experts a multiple of num_ranks and <= 4096,
 *     num_topk 1..32, num_tokens >= 0, num_nodes 1..num_ranks dividing
 *     num_ranks (node outputs are written only when num_tokens_per_node is
 *     non-NULL).  The scratch needed is
 *     4 * (128 + R * ceil(max(T,1) / 256) * (E + R + N)) bytes, N = num_nodes
 *     when node outputs are requested and 0 otherwise; a call that
 *     needs more than EP_LAYOUT_NOALLOC_SCRATCH_BYTES returns EP_ERR_CAPACITY
 *     and launches nothing (use ep_get_dispatch_layout instead).
 *   - status_out (device, nullable): if given, the kernel ORs its error bits
 *     into it (1 = a topk_idx value outside [-1, E) was skipped); the caller
 *     zeroes it.  If NULL, the error bits go to a word of the shared scratch
 *     that no caller can read and the next call clears: an out-of-range
 *     topk_idx value is then skipped silently.  Pass status_out whenever the
 *     routing is not known to be valid.
 *   - The first call on a device looks up the scratch array's device address
 *     (once per device, with that device current); make that first call before
 *     any stream capture.  Every call clears the counters it needs before its
 *     kernel runs, on `stream`.  All calls share the one array: calls whose
 *     kernels overlap on the GPU (other streams, other threads) race and give
 *     wrong results; order them on one stream. */
#define EP_LAYOUT_NOALLOC_SCRATCH_BYTES (1u << 20)
ep_status ep_get_dispatch_layout_noalloc(int32_t num_ranks, int32_t num_experts, int32_t num_topk,
                                         int32_t num_tokens, int32_t num_nodes, const int64_t* topk_idx,
                                         int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                                         uint8_t* is_token_in_rank, int32_t* num_tokens_per_node,
                                         uint8_t* is_token_in_node, uint32_t* status_out, void* stream);

/* ------------------------------------------------------------------------ */
/* Notify: count exchange, ragged offsets, channel prefix, positions          */
/* ([P1] 事件驱动调度的本质 / 高吞吐量模式; [P2] notify_dispatch steps 1-3)        */
/* ------------------------------------------------------------------------ */

/* The handle ("发货单", the shipping bill combine routes back with).  Every
 * member is a caller-allocated device array of the stated shape. */
typedef struct ep_dispatch_handle {
    int32_t* recv_count;            /* [R][R]  (d, s) = num_tokens_per_rank[s][d]         */
    int32_t* recv_offsets;          /* [R][R]  exclusive prefix over s of recv_count[d]   */
    int32_t* num_recv_tokens;       /* [R]     rows rank d receives                        */
    int32_t* rank_base;             /* [R+1]   exclusive prefix of num_recv_tokens         */
    int32_t* num_recv_per_expert;   /* [R][L]  pairs for local expert l of rank d          */
    int32_t* expert_offsets;        /* [R][L]  exclusive prefix over l                     */
    int32_t* perm_rank_base;        /* [R+1]   exclusive prefix over d of rank d's pairs   */
    int32_t* channel_prefix_matrix; /* [R][R][C] inclusive prefix over channels of the
                                       per-channel copy counts of (s, d)                  */
    int32_t* send_pos;              /* [R][T][R] row of (s,t) inside receiver d's block, -1 */
    int32_t* perm_pos;              /* [R][T][K] permuted row of pair (s,t,k), -1 if masked */
    int32_t* stage_base;            /* [R+1]   hierarchical only (else NULL): staging rows
                                       of home rank h start at stage_base[h]              */
    int32_t* stage_pos;             /* [R][T][N] hierarchical only (else NULL)             */
} ep_dispatch_handle;

/* Reads the layout (and topk_idx), fills the handle, and waits for the
 * receive counts ([P2] intranode_dispatch step 3, "CPU 同步等待 GPU 把接收计数写好"):
 *   host_num_recv_tokens     [R]   rows each rank receives;
 *   host_num_recv_per_expert [R*L] (nullable) pairs per local expert;
 *   host_totals              [3]   (nullable) total received rows (sum over d),
 *                                  total permuted rows (P), total staged rows.
 * These host values size the caller's receive buffers.  Receive order inside
 * rank d is (source s, token t) ascending; permuted order inside rank d is
 * (local expert, s, t, k).  The node pointers are required iff N > 1.
 *
 * No-wait form (host_num_recv_tokens, host_num_recv_per_expert and
 * host_totals all NULL): only the two kernels are enqueued; nothing waits on
 * the host, so the normal path (layout, notify, dispatch, permute, combine)
 * can be captured in a CUDA graph.  This departs from the pages' host wait:
 * the totals stay on the device (rank_base[R] received rows, perm_rank_base[R]
 * permuted rows, stage_base[R] staged rows), and until the next waiting
 * notify the later calls take their capacity arguments as the row bounds,
 * size their grids from them and read the actual counts from the handle on
 * the device.  Buffers sized for the worst case never overflow: received rows
 * <= R*T*min(K, R), permuted rows <= R*T*K (plus E*(alignment-1) with an
 * expert alignment), staged rows <= R*T*min(K, N).
 * Smaller buffers are allowed; rows past a capacity are not written and the
 * device status reports EP_ERR_CAPACITY (ep_ctx_check).  A topk_idx value
 * outside [-1, E) is likewise reported by ep_ctx_check. */
ep_status ep_notify_dispatch(ep_ctx* ctx, const int64_t* topk_idx,
                             const int32_t* num_tokens_per_expert,
                             const int32_t* num_tokens_per_rank, const uint8_t* is_token_in_rank,
                             const int32_t* num_tokens_per_node, const uint8_t* is_token_in_node,
                             const ep_dispatch_handle* handle, int32_t* host_num_recv_tokens,
                             int32_t* host_num_recv_per_expert, int32_t* host_totals, void* stream);

/* Layout and notify together ([P2] DeepEP v2: the notify warps compute the
 * layout on the fly instead of a separate get_dispatch_layout launch): the
 * layout outputs of ep_get_dispatch_layout are written (num_tokens_per_node /
 * is_token_in_node required iff N > 1, else NULL) and the handle is filled as
 * by ep_notify_dispatch, in two kernel launches instead of three (one kernel
 * computes the layout histograms, which are also notify's per-tile counts,
 * and the CTA completing the last source runs the offset scans).  Same
 * waiting and no-wait forms, same results. */
ep_status ep_layout_notify(ep_ctx* ctx, const int64_t* topk_idx, int32_t* num_tokens_per_expert,
                           int32_t* num_tokens_per_rank, uint8_t* is_token_in_rank,
                           int32_t* num_tokens_per_node, uint8_t* is_token_in_node,
                           const ep_dispatch_handle* handle, int32_t* host_num_recv_tokens,
                           int32_t* host_num_recv_per_expert, int32_t* host_totals, void* stream);

/* ------------------------------------------------------------------------ */
/* Dispatch scatter (v2 rank-level dedup) and local permute                 */
/* ([P2] dispatch 过程, v2 direct 模式 "同一 destination rank 只发一份";           */
/*  [P1] 高吞吐量模式 "本地置换（local permute）")                                 */
/* ------------------------------------------------------------------------ */

/* For each (s, t, d) with is_token_in_rank, writes row rank_base[d] +
 * send_pos[s][t][d] of:
 *   recv_x [rows][H] bf16 = x[s][t] (each source row read once);
 *   recv_src_rank, recv_src_idx [rows] int32 = (s, t);
 *   recv_topk_idx [rows][K] int32 = local expert id where expert k is on d, else -1;
 *   recv_topk_weights [rows][K] fp32 = the weight where expert k is on d, else 0.
 * recv_capacity_rows is the number of rows the recv_* arrays hold (must be
 * >= the total from the last waiting ep_notify_dispatch, else
 * EP_ERR_CAPACITY; after the no-wait form the check is made on the device). */
ep_status ep_dispatch(ep_ctx* ctx, const void* x, const int64_t* topk_idx,
                      const float* topk_weights, const ep_dispatch_handle* handle, void* recv_x,
                      int32_t* recv_src_rank, int32_t* recv_src_idx, int32_t* recv_topk_idx,
                      float* recv_topk_weights, int64_t recv_capacity_rows, void* stream);

/* Replicates each received row once per valid local expert into contiguous
 * per-expert blocks (the grouped-GEMM layout): permuted_x [P][H] bf16 at rows
 * perm_pos, perm_src_row [P] int32 = the recv_x row each came from.
 * Reads the recv_* arrays ep_dispatch wrote: the handle's rank_base[R] rows,
 * read on the device; num_recv_rows (> 0) is the most it may read (the recv
 * arrays' capacity, or the waiting notify's total). */
ep_status ep_permute(ep_ctx* ctx, const ep_dispatch_handle* handle, const void* recv_x,
                     const int32_t* recv_src_rank, const int32_t* recv_src_idx,
                     const int32_t* recv_topk_idx, int64_t num_recv_rows, void* permuted_x,
                     int32_t* perm_src_row, int64_t perm_capacity_rows, void* stream);

/* Fused dispatch: each token written once per valid top-k entry straight into
 * its permuted row (the expert-major blocks ep_permute produces), without the
 * per-rank receive buffer ([P2] DeepEP v2 direct 模式: the dispatch kernel's
 * epilogue arranges the data into the tensors the experts consume; this skips
 * recv_x).  permuted_x [P][H] bf16 equals ep_permute's output;
 * perm_src_token [P] int32 = s*T + t of each row; perm_weight [P] fp32
 * (nullable) = the entry's weight.  Needs the handle of ep_notify_dispatch. */
ep_status ep_dispatch_permuted(ep_ctx* ctx, const void* x, const int64_t* topk_idx,
                               const float* topk_weights, const ep_dispatch_handle* handle,
                               void* permuted_x, int32_t* perm_src_token, float* perm_weight,
                               int64_t perm_capacity_rows, void* stream);

/* ------------------------------------------------------------------------ */
/* FP8 rows for the normal path ([P2] 内存布局: a token's message carries x and  */
/* its scales; [P1] 低延迟模式: hidden states travel as FP8, combine stays BF16) */
/* ------------------------------------------------------------------------ */

/* Bytes of one FP8 row: H e4m3 codes, then H/128 fp32 scales, padded to 16. */
int64_t ep_fp8_row_bytes(int hidden);

/* Quantises every token of x [R][T][H] bf16 once into xq [R*T][fp8 row]:
 * per 128 channels scale = amax / 448 (fp32 division), code = e4m3
 * RNE-satfinite of x / scale (fp32 division); a zero scale keeps only the
 * sign.  Needs hidden % 128 == 0. */
ep_status ep_quantize_fp8(ep_ctx* ctx, const void* x, uint8_t* xq, void* stream);

/* ep_dispatch, ep_permute and ep_dispatch_permuted on FP8 rows (same metadata,
 * same row positions; recv_xq / permuted_xq hold FP8 rows). */
ep_status ep_dispatch_fp8(ep_ctx* ctx, const uint8_t* xq, const int64_t* topk_idx,
                          const float* topk_weights, const ep_dispatch_handle* handle,
                          uint8_t* recv_xq, int32_t* recv_src_rank, int32_t* recv_src_idx,
                          int32_t* recv_topk_idx, float* recv_topk_weights,
                          int64_t recv_capacity_rows, void* stream);
ep_status ep_permute_fp8(ep_ctx* ctx, const ep_dispatch_handle* handle, const uint8_t* recv_xq,
                         const int32_t* recv_src_rank, const int32_t* recv_src_idx,
                         const int32_t* recv_topk_idx, int64_t num_recv_rows, uint8_t* permuted_xq,
                         int32_t* perm_src_row, int64_t perm_capacity_rows, void* stream);
ep_status ep_dispatch_permuted_fp8(ep_ctx* ctx, const uint8_t* xq, const int64_t* topk_idx,
                                   const float* topk_weights, const ep_dispatch_handle* handle,
                                   uint8_t* permuted_xq, int32_t* perm_src_token, float* perm_weight,
                                   int64_t perm_capacity_rows, void* stream);

/* Quantise and dispatch in one pass: the bf16 tokens x [R][T][H] are
 * quantised (the rule of ep_quantize_fp8) and each FP8 row written straight
 * into its permuted rows ([P1] 低延迟模式: FP8 conversion fused into the send;
 * here for the normal path's expert-major layout).  permuted_xq,
 * perm_src_token and perm_weight equal those of ep_quantize_fp8 followed by
 * ep_dispatch_permuted_fp8 (padding bytes of a row excepted), without the
 * intermediate [R*T] FP8 rows. */
ep_status ep_dispatch_permuted_quant(ep_ctx* ctx, const void* x, const int64_t* topk_idx,
                                     const float* topk_weights, const ep_dispatch_handle* handle,
                                     uint8_t* permuted_xq, int32_t* perm_src_token, float* perm_weight,
                                     int64_t perm_capacity_rows, void* stream);
/* The same for the dispatch scatter's receive layout: recv_xq (FP8 rows) and
 * the recv_* metadata equal those of ep_quantize_fp8 followed by
 * ep_dispatch_fp8. */
ep_status ep_dispatch_quant(ep_ctx* ctx, const void* x, const int64_t* topk_idx, const float* topk_weights,
                            const ep_dispatch_handle* handle, uint8_t* recv_xq, int32_t* recv_src_rank,
                            int32_t* recv_src_idx, int32_t* recv_topk_idx, float* recv_topk_weights,
                            int64_t recv_capacity_rows, void* stream);

/* ------------------------------------------------------------------------ */
/* Combine ([P2] combine 过程; v2 "rank-level partial result ... epilogue 按    */
/* 不同 destination rank 做最终归约")                                             */
/* ------------------------------------------------------------------------ */

/* out[s][t] = bf16( sum over d ascending of ( sum over k ascending with
 * expert k on rank d of w[s][t][k] * y[perm_pos[s][t][k]] ) ): each rank
 * partial is an fp32 fused multiply-add chain, the partials are added in fp32
 * in rank order, the result is rounded to bf16 (nearest-even).  Tokens with no
 * valid entry get +0.  expert_out [P][H] bf16 is in the permuted layout.  No
 * host synchronisation. */
ep_status ep_combine(ep_ctx* ctx, const ep_dispatch_handle* handle, const void* expert_out,
                     int64_t num_perm_rows, const int64_t* topk_idx, const float* topk_weights,
                     void* out, void* stream);

/* ------------------------------------------------------------------------ */
/* Hierarchical (node, then rank) staging  ([P2] hybrid 模式; [P1] 零拷贝通信:   */
/* home rank = the GPU with the same index on the target node)               */
/* ------------------------------------------------------------------------ */

/* Stage A: one copy of x[s][t] per destination node n, into the staging rows
 * of home rank h = n*G + s % G (rows of a home rank ordered by (s, t)):
 * staging [stage rows][H] bf16, stage_src_rank / stage_src_idx [stage rows].
 * Stage B: each staged row is forwarded to every rank d of its node with
 * is_token_in_rank[s][t][d], at the same recv row as ep_dispatch, together
 * with the same recv metadata.  The result equals ep_dispatch's. */
ep_status ep_dispatch_hier(ep_ctx* ctx, const void* x, const int64_t* topk_idx,
                           const float* topk_weights, const ep_dispatch_handle* handle,
                           void* staging, int32_t* stage_src_rank, int32_t* stage_src_idx,
                           int64_t stage_capacity_rows, void* recv_x, int32_t* recv_src_rank,
                           int32_t* recv_src_idx, int32_t* recv_topk_idx,
                           float* recv_topk_weights, int64_t recv_capacity_rows, void* stream);

/* As ep_combine, grouped in three levels: rank partial (k ascending), node
 * partial (ranks of the node ascending), final (nodes ascending), all fp32. */
ep_status ep_combine_hier(ep_ctx* ctx, const ep_dispatch_handle* handle, const void* expert_out,
                          int64_t num_perm_rows, const int64_t* topk_idx,
                          const float* topk_weights, void* out, void* stream);

/* ------------------------------------------------------------------------ */
/* Low-latency mode ([P1] 低延迟模式; [P2] low-latency ping-pong; [P3] 2.2, 4.2) */
/* ------------------------------------------------------------------------ */

typedef struct ep_ll_buffer ep_ll_buffer;

/* Bytes of one message: a 16-byte header (source token index), H e4m3 codes,
 * H/128 fp32 scales, rounded up to 16. */
int64_t ep_ll_message_bytes(int hidden);

/* Bytes the two ping-pong buffers take ([P3] 2.2 get_low_latency_rdma_size_hint):
 * per buffer E*R*cap messages and E*R int32 count slots (padded to 16
 * bytes), rounded up to a multiple of 128.
 * Worst case by construction: every (expert, source) region holds `cap`. */
int64_t ep_ll_size_hint(int num_max_dispatch_tokens_per_rank, int hidden, int num_ranks,
                        int num_experts);

/* Allocates the two ping-pong buffers (count slots set to the empty sentinel
 * -1, [P2] "初始化计数器为 -1") on the current device.  cfg->hidden must be a
 * multiple of 128; cap = tokens per (expert, source) region, 1..4096. */
ep_status ep_ll_buffer_create(const ep_config* cfg, int cap, ep_ll_buffer** out);
void ep_ll_buffer_destroy(ep_ll_buffer* buf);

/* Limit of the receiver's count-slot waits, microseconds (default 100 000). */
ep_status ep_ll_set_wait_timeout_us(ep_ll_buffer* buf, int64_t us);

/* Signal-wait trace ([P1] 工程实践：模式选择与监控要点, the low-latency mode's
 * count-slot wait distribution): with wait_ns a caller-owned device array
 * [E][R] int64, every later ep_ll_recv writes, per (expert e, source s), the
 * nanoseconds from its receive CTA's start until that CTA had read the counts
 * it needs (the wait for the publisher included).  NULL stops the trace. */
ep_status ep_ll_set_wait_trace(ep_ll_buffer* buf, int64_t* wait_ns);

/* Sends the microbatch of tokens [t0, t0+n) of every source rank (n <= cap):
 * flips to the other ping-pong buffer, quantises each token once to e4m3 with
 * per-128-channel fp32 scales (scale = amax / 448, code = RNE-satfinite(x /
 * scale), a zero scale keeps only the sign), and writes one message per valid
 * (t, k) to slot `slot` of region (e*R + s) (address = base + (expert*R +
 * src_rank)*cap + slot, [P1] 低延迟模式).  The slot of (s, t, k) is the number
 * of earlier (t', k') of the same source and microbatch with the same expert;
 * it is written to slot_out [R][T][K] (rows t0..t0+n-1; -1 if masked).  After
 * the data of a source, every count slot count[e][s] of that source is
 * written, 0 included, with release ordering, so a visible count means its
 * data is in place.  Also resets the other buffer's count slots to -1. */
ep_status ep_ll_send(ep_ll_buffer* buf, const void* x, const int64_t* topk_idx, int t0, int n,
                     int32_t* slot_out, void* stream);

/* Receives the current buffer ([P3] 4.2): per (local expert, source) waits
 * (bounded) until the count slot leaves -1, then packs:
 *   packed_x [R][L][R*cap][H] uint8 e4m3, packed_scales [R][L][R*cap][H/128] fp32,
 *   packed_src_info [R][L][R*cap][2] int32 = (s, t),
 *   packed_recv_count [R][L] int32, layout_range [R][L][R][2] int32 = (begin, count)
 * with sources in ascending order inside each expert block.  A wait that runs
 * out records EP_ERR_TIMEOUT (ep_ll_check) and treats that source as empty. */
ep_status ep_ll_recv(ep_ll_buffer* buf, uint8_t* packed_x, float* packed_scales,
                     int32_t* packed_src_info, int32_t* packed_recv_count, int32_t* layout_range,
                     void* stream);

/* ep_ll_send followed by ep_ll_recv on the same stream (no host sync). */
ep_status ep_ll_dispatch(ep_ll_buffer* buf, const void* x, const int64_t* topk_idx, int t0, int n,
                         uint8_t* packed_x, float* packed_scales, int32_t* packed_src_info,
                         int32_t* packed_recv_count, int32_t* layout_range, int32_t* slot_out,
                         void* stream);

/* BF16 combine of the microbatch [t0, t0+n): out[s][t] = bf16( fp32 fma over
 * k ascending of w[s][t][k] * y_ll[d][l][begin(d,l,s) + slot(s,t,k)] ),
 * y_ll [R][L][R*cap][H] bf16 in the packed layout. */
ep_status ep_ll_combine(ep_ll_buffer* buf, const void* y_ll, const int64_t* topk_idx,
                        const float* topk_weights, const int32_t* slot,
                        const int32_t* layout_range, int t0, int n, void* out, void* stream);

/* Synchronises `stream`, reads and clears the buffer's status word. */
ep_status ep_ll_check(ep_ll_buffer* buf, void* stream);

/* Device pointer to the count slots [E][R] int32 of ping-pong buffer
 * `which` (0 or 1), and the index of the buffer the last send used. */
int32_t* ep_ll_count_slots(ep_ll_buffer* buf, int which);
int ep_ll_current_buffer(const ep_ll_buffer* buf);

#ifdef __cplusplus
}
#endif
#endif /* EP_GB300_H */
