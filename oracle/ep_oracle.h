/*
 * ep_oracle.h -- plain CPU oracle for MoE expert-parallel dispatch / combine.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg may load this library.  It shares no code with the CUDA
 * path and is deliberately slow and scalar: every function is the plain
 * definition of one step, in the order the method states it.
 *
 * Notation: R ranks, E experts (L = E / R per rank, expert e on rank e / L),
 * K top-k, T tokens per source rank, H hidden (bf16), C channels, N nodes
 * (G = R / N ranks per node, rank r on node r / G).  Arrays are row-major and
 * concatenated over ranks.  bf16 values travel as uint16_t bit patterns.
 *
 * Return value of every function: 0 on success, -1 on a bad argument,
 * -2 when topk_idx holds a value outside [-1, E).
 */
#ifndef EP_ORACLE_H
#define EP_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- number formats ---------------------------------------------------- */
float    orc_bf16_to_f32(uint16_t b);
uint16_t orc_f32_to_bf16(float f);          /* round to nearest, ties to even   */
uint16_t orc_f64_to_bf16(double v);         /* direct RNE from double           */
uint8_t  orc_e4m3_encode(float v);          /* OCP e4m3: RNE, saturate to +-448 */
float    orc_e4m3_decode(uint8_t code);
void     orc_e4m3_encode_array(const float* v, uint8_t* out, int64_t n);
/* per-128-channel block quantisation of one bf16 row (H % 128 == 0) */
void     orc_quantize_row(const uint16_t* x, int H, uint8_t* codes, float* scales);

/* ---- layout (get_dispatch_layout) -------------------------------------- */
int orc_layout(int R, int E, int K, int T, int N, const int64_t* topk_idx,
               int32_t* num_tokens_per_expert /*[R][E]*/, int32_t* num_tokens_per_rank /*[R][R]*/,
               uint8_t* is_token_in_rank /*[R][T][R]*/,
               int32_t* num_tokens_per_node /*[R][N] or NULL*/, uint8_t* is_token_in_node /*[R][T][N] or NULL*/);

/* ---- notify (counts exchange, offsets, channel prefix, send positions) --- */
int orc_notify(int R, int E, int T, int C,
               const int32_t* num_tokens_per_expert, const int32_t* num_tokens_per_rank,
               const uint8_t* is_token_in_rank,
               int32_t* recv_count /*[R][R] (d,s)*/, int32_t* num_recv_tokens /*[R]*/,
               int32_t* recv_offsets /*[R][R] (d,s)*/, int32_t* rank_base /*[R+1]*/,
               int32_t* num_recv_per_expert /*[R][L]*/, int32_t* expert_offsets /*[R][L]*/,
               int32_t* perm_rank_base /*[R+1]*/, int32_t* channel_prefix_matrix /*[R][R][C]*/,
               int32_t* send_pos /*[R][T][R]*/);

/* As orc_notify; every (d, l) block of the permuted layout takes its count
 * rounded up to a multiple of align rows (expert_offsets, perm_rank_base). */
int orc_notify_aligned(int R, int E, int T, int C, int align,
                       const int32_t* num_tokens_per_expert, const int32_t* num_tokens_per_rank,
                       const uint8_t* is_token_in_rank, int32_t* recv_count, int32_t* num_recv_tokens,
                       int32_t* recv_offsets, int32_t* rank_base, int32_t* num_recv_per_expert,
                       int32_t* expert_offsets, int32_t* perm_rank_base, int32_t* channel_prefix_matrix,
                       int32_t* send_pos);

/* ---- dispatch scatter (one copy per destination rank) ------------------- */
int orc_dispatch(int R, int E, int K, int T, int H,
                 const uint16_t* x, const int64_t* topk_idx, const float* topk_weights,
                 const int32_t* send_pos, const int32_t* rank_base,
                 uint16_t* recv_x, int32_t* recv_src_rank, int32_t* recv_src_idx,
                 int32_t* recv_topk_idx, float* recv_topk_weights);

/* ---- local permute: stable sort of the (s,t,k) pairs by (d, l, s, t, k) -- */
int orc_permute(int R, int E, int K, int T, int H, const int64_t* topk_idx,
                const uint16_t* recv_x, const int32_t* rank_base, const int32_t* send_pos,
                uint16_t* permuted_x /*[P][H]*/, int32_t* perm_src_row /*[P]*/,
                int32_t* perm_pos /*[R][T][K]*/);
/* Aligned blocks: padding rows get perm_src_row -1; rows = output rows or -1. */
int orc_permute_aligned(int R, int E, int K, int T, int H, int align, int64_t rows, const int64_t* topk_idx,
                        const uint16_t* recv_x, const int32_t* rank_base, const int32_t* send_pos,
                        uint16_t* permuted_x, int32_t* perm_src_row, int32_t* perm_pos);

/* ---- combine ------------------------------------------------------------ */
/* fp32 fmaf in the defined order: per destination rank d ascending, the rank
 * partial over k ascending; partials summed over d ascending; bf16 RNE. */
int orc_combine_ord32(int R, int E, int K, int T, int H, const uint16_t* expert_out,
                      const int32_t* perm_pos, const int64_t* topk_idx, const float* topk_weights,
                      uint16_t* out);
/* fp64 sum of all valid terms, rounded once to bf16. */
int orc_combine_ref64(int R, int E, int K, int T, int H, const uint16_t* expert_out,
                      const int32_t* perm_pos, const int64_t* topk_idx, const float* topk_weights,
                      uint16_t* out);

/* ---- low-latency mode ---------------------------------------------------- */
/* Send for the microbatch of tokens [t0, t0+n) of every source rank.
 * Region of (expert e, source s) = slots (e*R + s)*cap .. +cap-1.
 * reg_codes [E*R*cap][H], reg_scales [E*R*cap][H/128], reg_src [E*R*cap],
 * counts [E][R] (every pair written, 0 included), slot [R][T][K] (-1 masked;
 * only rows t0..t0+n-1 are written).  Returns -3 when a region overflows cap. */
int orc_ll_send(int R, int E, int K, int T, int H, int cap, int t0, int n,
                const uint16_t* x, const int64_t* topk_idx,
                uint8_t* reg_codes, float* reg_scales, int32_t* reg_src,
                int32_t* counts, int32_t* slot);
/* Receive + pack: packed_* [R][L][R*cap]..., packed_src_info [R][L][R*cap][2] = (s,t),
 * packed_recv_count [R][L], layout_range [R][L][R][2] = (begin, count). */
int orc_ll_pack(int R, int E, int H, int cap,
                const uint8_t* reg_codes, const float* reg_scales, const int32_t* reg_src,
                const int32_t* counts,
                uint8_t* packed_x, float* packed_scales, int32_t* packed_src_info,
                int32_t* packed_recv_count, int32_t* layout_range);
/* out rows t0..t0+n-1 of each rank: fp32 fmaf over k ascending; bf16 RNE. */
int orc_ll_combine(int R, int E, int K, int T, int H, int cap, int t0, int n,
                   const uint16_t* y_ll /*[R][L][R*cap][H]*/, const int64_t* topk_idx,
                   const float* topk_weights, const int32_t* slot, const int32_t* layout_range,
                   uint16_t* out /*[R][T][H]*/);
/* identity expert for LL: y = bf16_RNE(float(code) * scale) */
int orc_ll_dequant(int rows, int H, const uint8_t* codes, const float* scales, uint16_t* y);

/* ---- hierarchical (node, then rank) staging ----------------------------- */
/* Home rank of source s on node n: n*G + s % G.  Staging rows are grouped by
 * home rank ascending and ordered by (s, t) inside a home rank. */
int orc_hier_stage_pos(int R, int T, int N, const int32_t* num_tokens_per_node,
                       const uint8_t* is_token_in_node,
                       int32_t* stage_base /*[R+1]*/, int32_t* stage_pos /*[R][T][N]*/);
int orc_hier_stage_a(int R, int T, int H, int N, const uint16_t* x, const int32_t* stage_pos,
                     uint16_t* staging, int32_t* stage_src_rank, int32_t* stage_src_idx);
int orc_hier_stage_b(int R, int T, int H, int N, int num_stage_rows, const int32_t* stage_base,
                     const uint16_t* staging, const int32_t* stage_src_rank,
                     const int32_t* stage_src_idx, const uint8_t* is_token_in_rank,
                     const int32_t* send_pos, const int32_t* rank_base, uint16_t* recv_x);
/* rank partial (k ascending) -> node partial (ranks of the node ascending)
 * -> final (nodes ascending), fp32, bf16 RNE. */
int orc_combine_hier_ord32(int R, int E, int K, int T, int H, int N, const uint16_t* expert_out,
                           const int32_t* perm_pos, const int64_t* topk_idx,
                           const float* topk_weights, uint16_t* out);

/* ---- LL buffer size -------------------------------------------------------- */
int64_t orc_ll_message_bytes(int H);
int64_t orc_ll_size_hint(int num_max_dispatch_tokens_per_rank, int hidden, int num_ranks,
                         int num_experts);

#ifdef __cplusplus
}
#endif
#endif
