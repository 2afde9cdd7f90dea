/*
 * ep_oracle.c -- plain CPU oracle for MoE expert-parallel dispatch / combine.
 *
 * TEST INFRASTRUCTURE ONLY (tests, smoke check and the bench's CPU-baseline
 * leg).  Nothing here is shared with the CUDA path.  Each function is the
 * scalar definition of one step of the method described on the pages
 * "DeepEP 学习笔记" (sections "dispatch 前：全局布局与通知", "dispatch 过程",
 * "combine 过程", "DeepEP v2 / direct 模式", "hybrid 模式"), "事件驱动 EP 内核的调度
 * 策略与零拷贝通信" (sections "高吞吐量模式" and "低延迟模式") and "DeepSeek DeepEP
 * 探索：低延迟分发" (sections 2.2 and 4.2).
 *
 * Build: gcc -O2 -ffp-contract=off -std=c11 -shared -fPIC (no fast-math: the
 * float divisions and fmaf calls must be the IEEE-754 operations).
 */
#include "ep_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ======================================================================== */
/* Number formats                                                           */
/* ======================================================================== */

float orc_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* bf16 keeps the top 16 bits of an fp32; round the dropped 16 bits to the
 * nearest value, ties to the even kept pattern. */
uint16_t orc_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0) /* NaN */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lower = u & 0xFFFFu;
    uint32_t upper = u >> 16;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

/* round-half-even of a non-negative double that is exactly representable */
static double rne_nonneg(double q) {
    double fl = floor(q);
    double diff = q - fl;
    if (diff > 0.5) return fl + 1.0;
    if (diff < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* Direct double -> bf16 (8 significant bits, exponent range of fp32). */
uint16_t orc_f64_to_bf16(double v) {
    if (isnan(v)) return 0x7FC0u;
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);             /* a = m * 2^e, m in [0.5, 1) */
    int E = e - 1;            /* a in [2^E, 2^(E+1)) */
    if (E < -126) E = -126;   /* subnormal: fixed quantum 2^-133 */
    double quantum = ldexp(1.0, E - 7);
    double q = rne_nonneg(a / quantum); /* exact scaling by a power of two; q <= 256 */
    double r = q * quantum;
    if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u); /* overflow -> inf */
    float rf = (float)r;      /* exact: r has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &rf, 4);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFFu));
}

/* OCP 8-bit floating point, E4M3 variant: 1 sign bit, 4 exponent bits (bias
 * 7), 3 mantissa bits; no infinities; S.1111.111 is NaN, so the largest
 * finite magnitude is 1.75 * 2^8 = 448; subnormals are m * 2^-9.  Rounding is
 * to nearest, ties to even; magnitudes at or above 448 saturate to 448. */
uint8_t orc_e4m3_encode(float v) {
    uint32_t u;
    memcpy(&u, &v, 4);
    uint8_t sign = (u >> 31) ? 0x80u : 0x00u;
    if (isnan(v)) return (uint8_t)(sign | 0x7Fu);
    double a = fabs((double)v);
    if (a >= 448.0) return (uint8_t)(sign | 0x7Eu);
    if (a < ldexp(1.0, -6)) {
        /* subnormal range; q == 8 carries into the smallest normal (0x08) */
        double q = rne_nonneg(a / ldexp(1.0, -9));
        return (uint8_t)(sign | (uint8_t)q);
    }
    int e;
    frexp(a, &e);
    int E = e - 1;                                  /* -6 .. 8 */
    double frac = a / ldexp(1.0, E) - 1.0;          /* [0, 1), exact */
    double q = rne_nonneg(frac * 8.0);              /* 0 .. 8 */
    if (q == 8.0) { q = 0.0; E += 1; }
    if (E > 8 || (E == 8 && q > 6.0)) return (uint8_t)(sign | 0x7Eu);
    return (uint8_t)(sign | (uint8_t)(((E + 7) << 3) | (int)q));
}

float orc_e4m3_decode(uint8_t c) {
    int s = c >> 7, ex = (c >> 3) & 0xF, m = c & 7;
    double v;
    if (ex == 0xF && m == 7) return NAN;
    if (ex == 0) v = m * ldexp(1.0, -9);
    else v = (1.0 + m / 8.0) * ldexp(1.0, ex - 7);
    return (float)(s ? -v : v);
}

void orc_e4m3_encode_array(const float* v, uint8_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(v[i]);
}

/* Per 128-channel block: amax = max |x|, scale = amax / 448 (fp32 division),
 * code = e4m3(x / scale) (fp32 division).  A zero scale keeps only the sign. */
void orc_quantize_row(const uint16_t* x, int H, uint8_t* codes, float* scales) {
    for (int b = 0; b < H / 128; ++b) {
        float amax = 0.0f;
        for (int i = 0; i < 128; ++i) {
            float a = fabsf(orc_bf16_to_f32(x[b * 128 + i]));
            if (a > amax) amax = a;
        }
        volatile float scale = amax / 448.0f;
        scales[b] = scale;
        for (int i = 0; i < 128; ++i) {
            float xv = orc_bf16_to_f32(x[b * 128 + i]);
            if (scale == 0.0f) {
                codes[b * 128 + i] = signbit(xv) ? 0x80u : 0x00u;
            } else {
                volatile float q = xv / scale;
                codes[b * 128 + i] = orc_e4m3_encode(q);
            }
        }
    }
}

/* ======================================================================== */
/* Layout: get_dispatch_layout                                              */
/* ======================================================================== */

static int check_shape(int R, int E, int K, int T) {
    if (R <= 0 || E <= 0 || K <= 0 || T < 0) return -1;
    if (E % R != 0) return -1;
    return 0;
}

int orc_layout(int R, int E, int K, int T, int N, const int64_t* topk_idx,
               int32_t* ntpe, int32_t* ntpr, uint8_t* itir, int32_t* ntpn, uint8_t* itin) {
    if (check_shape(R, E, K, T)) return -1;
    int use_nodes = (ntpn != NULL && itin != NULL && N > 0);
    if (use_nodes && R % N != 0) return -1;
    const int L = E / R;
    const int G = use_nodes ? R / N : 1;
    memset(ntpe, 0, sizeof(int32_t) * (size_t)R * E);
    memset(ntpr, 0, sizeof(int32_t) * (size_t)R * R);
    memset(itir, 0, (size_t)R * T * R);
    if (use_nodes) {
        memset(ntpn, 0, sizeof(int32_t) * (size_t)R * N);
        memset(itin, 0, (size_t)R * T * N);
    }
    int status = 0;
    for (int s = 0; s < R; ++s)
        for (int t = 0; t < T; ++t) {
            const int64_t* row = topk_idx + ((int64_t)s * T + t) * K;
            uint8_t* in_rank = itir + ((int64_t)s * T + t) * R;
            for (int k = 0; k < K; ++k) {
                int64_t e = row[k];
                if (e == -1) continue;
                if (e < -1 || e >= E) { status = -2; continue; }
                ntpe[s * E + e] += 1;
                in_rank[e / L] = 1;
                if (use_nodes) itin[((int64_t)s * T + t) * N + (e / L) / G] = 1;
            }
            for (int d = 0; d < R; ++d) ntpr[s * R + d] += in_rank[d];
            if (use_nodes)
                for (int n = 0; n < N; ++n) ntpn[s * N + n] += itin[((int64_t)s * T + t) * N + n];
        }
    return status;
}

/* ======================================================================== */
/* Notify                                                                   */
/* ======================================================================== */

int orc_notify(int R, int E, int T, int C, const int32_t* ntpe, const int32_t* ntpr,
               const uint8_t* itir, int32_t* recv_count, int32_t* num_recv_tokens,
               int32_t* recv_offsets, int32_t* rank_base, int32_t* num_recv_per_expert,
               int32_t* expert_offsets, int32_t* perm_rank_base, int32_t* cpm,
               int32_t* send_pos) {
    return orc_notify_aligned(R, E, T, C, 1, ntpe, ntpr, itir, recv_count, num_recv_tokens, recv_offsets,
                              rank_base, num_recv_per_expert, expert_offsets, perm_rank_base, cpm, send_pos);
}

/* round n up to a multiple of a (a >= 1) */
static int32_t round_up(int32_t n, int a) { return (n + a - 1) / a * a; }

int orc_notify_aligned(int R, int E, int T, int C, int align, const int32_t* ntpe, const int32_t* ntpr,
                       const uint8_t* itir, int32_t* recv_count, int32_t* num_recv_tokens,
                       int32_t* recv_offsets, int32_t* rank_base, int32_t* num_recv_per_expert,
                       int32_t* expert_offsets, int32_t* perm_rank_base, int32_t* cpm,
                       int32_t* send_pos) {
    if (R <= 0 || E <= 0 || E % R != 0 || T < 0 || C <= 0 || align < 1) return -1;
    const int L = E / R;
    /* all-gather of the per-peer counts, seen from each receiver d */
    for (int d = 0; d < R; ++d)
        for (int s = 0; s < R; ++s) recv_count[d * R + s] = ntpr[s * R + d];
    /* receiver totals and the exclusive prefix over sources */
    for (int d = 0; d < R; ++d) {
        int32_t acc = 0;
        for (int s = 0; s < R; ++s) {
            recv_offsets[d * R + s] = acc;
            acc += recv_count[d * R + s];
        }
        num_recv_tokens[d] = acc;
    }
    rank_base[0] = 0;
    for (int d = 0; d < R; ++d) rank_base[d + 1] = rank_base[d] + num_recv_tokens[d];
    /* per local expert totals and offsets; with an expert alignment a > 1
     * every expert's block takes its count rounded up to a multiple of a rows
     * (the tail rows are padding), so every block starts at a multiple of a */
    perm_rank_base[0] = 0;
    for (int d = 0; d < R; ++d) {
        int32_t acc = 0;
        for (int l = 0; l < L; ++l) {
            int32_t n = 0;
            for (int s = 0; s < R; ++s) n += ntpe[s * E + d * L + l];
            num_recv_per_expert[d * L + l] = n;
            expert_offsets[d * L + l] = acc;
            acc += round_up(n, align);
        }
        perm_rank_base[d + 1] = perm_rank_base[d] + acc;
    }
    /* channel c owns tokens [c*ct, min(T,(c+1)*ct)), ct = ceil(T / C); the
     * matrix holds the inclusive prefix over channels of per-channel counts */
    const int ct = (T + C - 1) / C;
    for (int s = 0; s < R; ++s)
        for (int d = 0; d < R; ++d) {
            int32_t acc = 0;
            for (int c = 0; c < C; ++c) {
                int lo = c * ct, hi = (c + 1) * ct;
                if (hi > T) hi = T;
                for (int t = lo; t < hi; ++t) acc += itir[((int64_t)s * T + t) * R + d];
                cpm[((int64_t)s * R + d) * C + c] = acc;
            }
        }
    /* send position: the source's offset at the receiver plus the number of
     * earlier tokens of the same source bound to the same receiver */
    for (int s = 0; s < R; ++s)
        for (int d = 0; d < R; ++d) {
            int32_t running = 0;
            for (int t = 0; t < T; ++t) {
                int64_t i = ((int64_t)s * T + t) * R + d;
                if (itir[i]) send_pos[i] = recv_offsets[d * R + s] + running++;
                else send_pos[i] = -1;
            }
        }
    return 0;
}

/* ======================================================================== */
/* Dispatch scatter                                                         */
/* ======================================================================== */

int orc_dispatch(int R, int E, int K, int T, int H, const uint16_t* x, const int64_t* topk_idx,
                 const float* topk_weights, const int32_t* send_pos, const int32_t* rank_base,
                 uint16_t* recv_x, int32_t* recv_src_rank, int32_t* recv_src_idx,
                 int32_t* recv_topk_idx, float* recv_topk_weights) {
    if (check_shape(R, E, K, T) || H <= 0) return -1;
    const int L = E / R;
    for (int s = 0; s < R; ++s)
        for (int t = 0; t < T; ++t)
            for (int d = 0; d < R; ++d) {
                int32_t p = send_pos[((int64_t)s * T + t) * R + d];
                if (p < 0) continue;
                int64_t row = (int64_t)rank_base[d] + p;
                memcpy(recv_x + row * H, x + ((int64_t)s * T + t) * H, sizeof(uint16_t) * (size_t)H);
                recv_src_rank[row] = s;
                recv_src_idx[row] = t;
                for (int k = 0; k < K; ++k) {
                    int64_t e = topk_idx[((int64_t)s * T + t) * K + k];
                    if (e >= 0 && e < E && e / L == d) {
                        recv_topk_idx[row * K + k] = (int32_t)(e - (int64_t)d * L);
                        recv_topk_weights[row * K + k] = topk_weights[((int64_t)s * T + t) * K + k];
                    } else {
                        recv_topk_idx[row * K + k] = -1;
                        recv_topk_weights[row * K + k] = 0.0f;
                    }
                }
            }
    return 0;
}

/* ======================================================================== */
/* Permute                                                                  */
/* ======================================================================== */

typedef struct { int32_t d, l, s, t, k; } pair_t;

static int pair_cmp(const void* a, const void* b) {
    const pair_t* p = (const pair_t*)a;
    const pair_t* q = (const pair_t*)b;
    if (p->d != q->d) return p->d < q->d ? -1 : 1;
    if (p->l != q->l) return p->l < q->l ? -1 : 1;
    if (p->s != q->s) return p->s < q->s ? -1 : 1;
    if (p->t != q->t) return p->t < q->t ? -1 : 1;
    if (p->k != q->k) return p->k < q->k ? -1 : 1;
    return 0;
}

int orc_permute(int R, int E, int K, int T, int H, const int64_t* topk_idx, const uint16_t* recv_x,
                const int32_t* rank_base, const int32_t* send_pos, uint16_t* permuted_x,
                int32_t* perm_src_row, int32_t* perm_pos) {
    return orc_permute_aligned(R, E, K, T, H, 1, -1, topk_idx, recv_x, rank_base, send_pos, permuted_x,
                               perm_src_row, perm_pos);
}

/* As orc_permute, each (d, l) block taking its pair count rounded up to a
 * multiple of align rows: pairs keep their (d, l, s, t, k) order, the block
 * of (d, l) starts at the sum of the rounded counts of the blocks before it,
 * and padding rows get perm_src_row = -1 (permuted_x rows left as they are).
 * rows = the number of rows the outputs hold (checked), or -1 to skip. */
int orc_permute_aligned(int R, int E, int K, int T, int H, int align, int64_t rows, const int64_t* topk_idx,
                        const uint16_t* recv_x, const int32_t* rank_base, const int32_t* send_pos,
                        uint16_t* permuted_x, int32_t* perm_src_row, int32_t* perm_pos) {
    if (check_shape(R, E, K, T) || H <= 0 || align < 1) return -1;
    const int L = E / R;
    int64_t P = 0;
    for (int64_t i = 0; i < (int64_t)R * T * K; ++i)
        if (topk_idx[i] >= 0 && topk_idx[i] < E) ++P;
    pair_t* pairs = (pair_t*)malloc(sizeof(pair_t) * (size_t)(P > 0 ? P : 1));
    if (!pairs) return -1;
    int64_t n = 0;
    for (int s = 0; s < R; ++s)
        for (int t = 0; t < T; ++t)
            for (int k = 0; k < K; ++k) {
                int64_t i = ((int64_t)s * T + t) * K + k;
                int64_t e = topk_idx[i];
                perm_pos[i] = -1;
                if (e < 0 || e >= E) continue;
                pair_t p = {(int32_t)(e / L), (int32_t)(e % L), s, t, k};
                pairs[n++] = p;
            }
    qsort(pairs, (size_t)n, sizeof(pair_t), pair_cmp);
    /* walk the sorted pairs block by block: a block is a run of equal (d, l);
     * empty blocks take no rows, so only the runs present advance the row */
    int64_t row = 0;
    for (int64_t i = 0; i < n;) {
        int64_t j = i;
        while (j < n && pairs[j].d == pairs[i].d && pairs[j].l == pairs[i].l) ++j;
        const int64_t cnt = j - i, padded = (cnt + align - 1) / align * align;
        if (rows >= 0 && row + padded > rows) {
            free(pairs);
            return -1;
        }
        for (int64_t q = 0; q < cnt; ++q) {
            const pair_t* p = &pairs[i + q];
            int32_t sp = send_pos[((int64_t)p->s * T + p->t) * R + p->d];
            int64_t src = (int64_t)rank_base[p->d] + sp;
            memcpy(permuted_x + (row + q) * H, recv_x + src * H, sizeof(uint16_t) * (size_t)H);
            perm_src_row[row + q] = (int32_t)src;
            perm_pos[((int64_t)p->s * T + p->t) * K + p->k] = (int32_t)(row + q);
        }
        for (int64_t q = cnt; q < padded; ++q) perm_src_row[row + q] = -1;
        row += padded;
        i = j;
    }
    free(pairs);
    if (rows >= 0 && row != rows) return -1;
    return 0;
}

/* ======================================================================== */
/* Combine                                                                  */
/* ======================================================================== */

int orc_combine_ord32(int R, int E, int K, int T, int H, const uint16_t* y, const int32_t* perm_pos,
                      const int64_t* topk_idx, const float* w, uint16_t* out) {
    if (check_shape(R, E, K, T) || H <= 0) return -1;
    const int L = E / R;
    for (int s = 0; s < R; ++s)
        for (int t = 0; t < T; ++t) {
            const int64_t tok = (int64_t)s * T + t;
            for (int j = 0; j < H; ++j) {
                float final_sum = 0.0f;
                for (int d = 0; d < R; ++d) {
                    int has = 0;
                    float partial = 0.0f;
                    for (int k = 0; k < K; ++k) {
                        int64_t e = topk_idx[tok * K + k];
                        if (e < 0 || e >= E || e / L != d) continue;
                        float yv = orc_bf16_to_f32(y[(int64_t)perm_pos[tok * K + k] * H + j]);
                        partial = fmaf(w[tok * K + k], yv, partial);
                        has = 1;
                    }
                    if (has) {
                        volatile float acc = final_sum + partial;
                        final_sum = acc;
                    }
                }
                out[tok * H + j] = orc_f32_to_bf16(final_sum);
            }
        }
    return 0;
}

int orc_combine_ref64(int R, int E, int K, int T, int H, const uint16_t* y, const int32_t* perm_pos,
                      const int64_t* topk_idx, const float* w, uint16_t* out) {
    if (check_shape(R, E, K, T) || H <= 0) return -1;
    for (int64_t tok = 0; tok < (int64_t)R * T; ++tok)
        for (int j = 0; j < H; ++j) {
            double acc = 0.0;
            for (int k = 0; k < K; ++k) {
                int64_t e = topk_idx[tok * K + k];
                if (e < 0 || e >= E) continue;
                acc += (double)w[tok * K + k] *
                       (double)orc_bf16_to_f32(y[(int64_t)perm_pos[tok * K + k] * H + j]);
            }
            out[tok * H + j] = orc_f64_to_bf16(acc);
        }
    return 0;
}

/* ======================================================================== */
/* Low-latency mode                                                         */
/* ======================================================================== */

int64_t orc_ll_message_bytes(int H) {
    /* 16-byte header (source token index + padding), H fp8 codes, H/128 fp32
     * scales, rounded up to 16 bytes */
    int64_t b = 16 + (int64_t)H + (int64_t)(H / 128) * 4;
    return (b + 15) / 16 * 16;
}

int64_t orc_ll_size_hint(int cap, int H, int R, int E) {
    /* two ping-pong buffers, each: E*R*cap messages + E*R int32 count slots
     * (padded to 16 bytes), rounded up to a multiple of 128 bytes */
    int64_t counts = ((int64_t)E * R * 4 + 15) / 16 * 16;
    int64_t one = (int64_t)E * R * cap * orc_ll_message_bytes(H) + counts;
    one = (one + 127) / 128 * 128;
    return 2 * one;
}

int orc_ll_send(int R, int E, int K, int T, int H, int cap, int t0, int n, const uint16_t* x,
                const int64_t* topk_idx, uint8_t* reg_codes, float* reg_scales, int32_t* reg_src,
                int32_t* counts, int32_t* slot) {
    if (check_shape(R, E, K, T) || H <= 0 || H % 128 != 0 || cap <= 0) return -1;
    if (t0 < 0 || n < 0 || t0 + n > T || n > cap) return -1;
    const int S = H / 128;
    uint8_t* codes = (uint8_t*)malloc((size_t)H);
    float* scales = (float*)malloc(sizeof(float) * (size_t)S);
    int32_t* running = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    if (!codes || !scales || !running) { free(codes); free(scales); free(running); return -1; }
    int status = 0;
    for (int s = 0; s < R; ++s) {
        memset(running, 0, sizeof(int32_t) * (size_t)E);
        /* (t, k) in lexicographic order: the slot is the number of earlier
         * entries of the same source bound to the same expert */
        for (int t = t0; t < t0 + n; ++t) {
            const int64_t tok = (int64_t)s * T + t;
            orc_quantize_row(x + tok * H, H, codes, scales);
            for (int k = 0; k < K; ++k) {
                int64_t e = topk_idx[tok * K + k];
                if (e == -1) { slot[tok * K + k] = -1; continue; }
                if (e < -1 || e >= E) { slot[tok * K + k] = -1; status = -2; continue; }
                int32_t sl = running[e]++;
                slot[tok * K + k] = sl;
                if (sl >= cap) { status = -3; continue; }
                /* addr = base + (expert_id * num_ranks + src_rank) * chunk + slot */
                int64_t m = ((int64_t)e * R + s) * cap + sl;
                memcpy(reg_codes + m * H, codes, (size_t)H);
                memcpy(reg_scales + m * S, scales, sizeof(float) * (size_t)S);
                reg_src[m] = t;
            }
        }
        /* every (expert, source) count slot is written, zero included */
        for (int e = 0; e < E; ++e) counts[(int64_t)e * R + s] = running[e];
    }
    free(codes);
    free(scales);
    free(running);
    return status;
}

int orc_ll_pack(int R, int E, int H, int cap, const uint8_t* reg_codes, const float* reg_scales,
                const int32_t* reg_src, const int32_t* counts, uint8_t* packed_x,
                float* packed_scales, int32_t* packed_src_info, int32_t* packed_recv_count,
                int32_t* layout_range) {
    if (R <= 0 || E <= 0 || E % R != 0 || H <= 0 || H % 128 != 0 || cap <= 0) return -1;
    const int L = E / R, S = H / 128;
    const int64_t per_expert = (int64_t)R * cap;
    for (int d = 0; d < R; ++d)
        for (int l = 0; l < L; ++l) {
            const int e = d * L + l;
            int32_t begin = 0;
            for (int s = 0; s < R; ++s) {
                int32_t c = counts[(int64_t)e * R + s];
                if (c < 0 || c > cap) return -3;
                int64_t lr = (((int64_t)d * L + l) * R + s) * 2;
                layout_range[lr] = begin;
                layout_range[lr + 1] = c;
                for (int i = 0; i < c; ++i) {
                    int64_t m = ((int64_t)e * R + s) * cap + i;
                    int64_t p = ((int64_t)d * L + l) * per_expert + begin + i;
                    memcpy(packed_x + p * H, reg_codes + m * H, (size_t)H);
                    memcpy(packed_scales + p * S, reg_scales + m * S, sizeof(float) * (size_t)S);
                    packed_src_info[p * 2] = s;
                    packed_src_info[p * 2 + 1] = reg_src[m];
                }
                begin += c;
            }
            packed_recv_count[d * L + l] = begin;
        }
    return 0;
}

int orc_ll_dequant(int rows, int H, const uint8_t* codes, const float* scales, uint16_t* y) {
    if (rows < 0 || H <= 0 || H % 128 != 0) return -1;
    const int S = H / 128;
    for (int64_t r = 0; r < rows; ++r)
        for (int j = 0; j < H; ++j) {
            volatile float v = orc_e4m3_decode(codes[r * H + j]) * scales[r * S + j / 128];
            y[r * H + j] = orc_f32_to_bf16(v);
        }
    return 0;
}

int orc_ll_combine(int R, int E, int K, int T, int H, int cap, int t0, int n, const uint16_t* y_ll,
                   const int64_t* topk_idx, const float* w, const int32_t* slot,
                   const int32_t* layout_range, uint16_t* out) {
    if (check_shape(R, E, K, T) || H <= 0 || cap <= 0) return -1;
    if (t0 < 0 || n < 0 || t0 + n > T) return -1;
    const int L = E / R;
    const int64_t per_expert = (int64_t)R * cap;
    for (int s = 0; s < R; ++s)
        for (int t = t0; t < t0 + n; ++t) {
            const int64_t tok = (int64_t)s * T + t;
            for (int j = 0; j < H; ++j) {
                float acc = 0.0f;
                for (int k = 0; k < K; ++k) {
                    int64_t e = topk_idx[tok * K + k];
                    if (e < 0 || e >= E) continue;
                    int d = (int)(e / L), l = (int)(e % L);
                    int32_t begin = layout_range[(((int64_t)d * L + l) * R + s) * 2];
                    int64_t row = ((int64_t)d * L + l) * per_expert + begin + slot[tok * K + k];
                    acc = fmaf(w[tok * K + k], orc_bf16_to_f32(y_ll[row * H + j]), acc);
                }
                out[tok * H + j] = orc_f32_to_bf16(acc);
            }
        }
    return 0;
}

/* ======================================================================== */
/* Hierarchical staging                                                     */
/* ======================================================================== */

int orc_hier_stage_pos(int R, int T, int N, const int32_t* ntpn, const uint8_t* itin,
                       int32_t* stage_base, int32_t* stage_pos) {
    if (R <= 0 || N <= 0 || R % N != 0 || T < 0) return -1;
    const int G = R / N;
    for (int64_t i = 0; i < (int64_t)R * T * N; ++i) stage_pos[i] = -1;
    int32_t acc = 0;
    for (int h = 0; h < R; ++h) {
        stage_base[h] = acc;
        const int n = h / G;
        /* sources whose home rank on node n is h, ascending, then tokens */
        for (int s = 0; s < R; ++s) {
            if (s % G != h % G) continue;
            for (int t = 0; t < T; ++t) {
                int64_t i = ((int64_t)s * T + t) * N + n;
                if (itin[i]) stage_pos[i] = acc++;
            }
        }
        (void)ntpn;
    }
    stage_base[R] = acc;
    return 0;
}

int orc_hier_stage_a(int R, int T, int H, int N, const uint16_t* x, const int32_t* stage_pos,
                     uint16_t* staging, int32_t* stage_src_rank, int32_t* stage_src_idx) {
    if (R <= 0 || N <= 0 || T < 0 || H <= 0) return -1;
    for (int s = 0; s < R; ++s)
        for (int t = 0; t < T; ++t)
            for (int n = 0; n < N; ++n) {
                int32_t p = stage_pos[((int64_t)s * T + t) * N + n];
                if (p < 0) continue;
                memcpy(staging + (int64_t)p * H, x + ((int64_t)s * T + t) * H,
                       sizeof(uint16_t) * (size_t)H);
                stage_src_rank[p] = s;
                stage_src_idx[p] = t;
            }
    return 0;
}

int orc_hier_stage_b(int R, int T, int H, int N, int num_stage_rows, const int32_t* stage_base,
                     const uint16_t* staging, const int32_t* stage_src_rank,
                     const int32_t* stage_src_idx, const uint8_t* itir, const int32_t* send_pos,
                     const int32_t* rank_base, uint16_t* recv_x) {
    if (R <= 0 || N <= 0 || R % N != 0 || H <= 0) return -1;
    const int G = R / N;
    int h = 0;
    for (int32_t i = 0; i < num_stage_rows; ++i) {
        while (h + 1 <= R && stage_base[h + 1] <= i) ++h; /* home rank of row i */
        const int n = h / G;
        const int s = stage_src_rank[i], t = stage_src_idx[i];
        for (int d = n * G; d < (n + 1) * G; ++d) {
            int64_t q = ((int64_t)s * T + t) * R + d;
            if (!itir[q]) continue;
            memcpy(recv_x + ((int64_t)rank_base[d] + send_pos[q]) * H, staging + (int64_t)i * H,
                   sizeof(uint16_t) * (size_t)H);
        }
    }
    return 0;
}

int orc_combine_hier_ord32(int R, int E, int K, int T, int H, int N, const uint16_t* y,
                           const int32_t* perm_pos, const int64_t* topk_idx, const float* w,
                           uint16_t* out) {
    if (check_shape(R, E, K, T) || H <= 0 || N <= 0 || R % N != 0) return -1;
    const int L = E / R, G = R / N;
    for (int64_t tok = 0; tok < (int64_t)R * T; ++tok)
        for (int j = 0; j < H; ++j) {
            float final_sum = 0.0f;
            for (int n = 0; n < N; ++n) {
                int node_has = 0;
                float node_sum = 0.0f;
                for (int d = n * G; d < (n + 1) * G; ++d) {
                    int has = 0;
                    float partial = 0.0f;
                    for (int k = 0; k < K; ++k) {
                        int64_t e = topk_idx[tok * K + k];
                        if (e < 0 || e >= E || e / L != d) continue;
                        float yv = orc_bf16_to_f32(y[(int64_t)perm_pos[tok * K + k] * H + j]);
                        partial = fmaf(w[tok * K + k], yv, partial);
                        has = 1;
                    }
                    if (has) {
                        volatile float a = node_sum + partial;
                        node_sum = a;
                        node_has = 1;
                    }
                }
                if (node_has) {
                    volatile float a = final_sum + node_sum;
                    final_sum = a;
                }
            }
            out[tok * H + j] = orc_f32_to_bf16(final_sum);
        }
    return 0;
}
