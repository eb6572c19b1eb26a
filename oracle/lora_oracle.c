/*
 * lora_oracle.c -- plain, slow fp64 CPU oracle for the heterogeneous
 * multi-LoRA linear layer.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or calls
 * this file: only the tests, the package's smoke check and the benchmark's
 * CPU-baseline leg do. It shares no code, header, table or helper with the
 * CUDA implementation.
 *
 * What it computes (the plain definition, written out as loops):
 *
 *   Y[t,n] = sum_k X[t,k] * W[n,k]
 *          + ( ids[t] >= 0 ? s_i * sum_j ( sum_k X[t,k] * A_i[k,j] ) * B_i[j,n] : 0 )
 *   with i = ids[t], s_i = alpha_i / r_i.
 *
 * Sources:
 *  - "LoRA-Land: 将大模型变成操作系统..." (blog), section 核心实现解析 /
 *    2. 多 LoRA 批处理调度: the base weight is shared and unchanged; each group of
 *    requests adds its own A,B correction, and X@A is formed first as a
 *    low-dimensional intermediate and then multiplied by B. The printed
 *    equation is garbled (its transposes do not type-check); the row-token
 *    reading Y = X W^T + s (X A) B with A d_in x r and B r x d_out is used.
 *  - "多 LoRA 热插拔: 一模型服多租户" (vLLM tutorial), section "LoRA 速览": the
 *    base weight is untouched and a low-rank side branch is added per linear
 *    layer (W'x = Wx + BAx, the same map in column-vector convention).
 *  - same tutorial, section "按请求切换 LoRA": a request with no adapter runs
 *    the pure base model (ids[t] = -1 here).
 *  - icman.com.cn Multi-LoRA article, section 2.1 (共享基座动态挂载 adapter):
 *    the "dynamic batching" mode picks each sample's low-rank matrices and adds
 *    the branch back onto the main path; the "merge" mode materialises
 *    W + BA first. Both compute the same result.
 *  - same article, section 3.2: alpha "controls the scaling" and is usually
 *    2*rank; the scale is read as s = alpha / rank (the rank the adapter was
 *    loaded with).
 *  - same article, section 4.1: an id that names no loaded adapter is an
 *    error (strict mode), never a silent fall-back to the base output.
 *
 * Inputs are bfloat16 bit patterns (uint16); every value is widened exactly to
 * double, all sums are in double, and the output is double (no rounding).
 *
 * Segments ("Grouped Multi-LoRA Execution", blog section 2: the batch is
 * grouped by LoRA ID and each group is run contiguously): order is the stable
 * ascending sort of token indices by id (ties keep token order), so the
 * base-only tokens (id -1) come first as a block of n_base tokens; every
 * maximal run of one id >= 0 in that order is one segment.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_BAD_ADAPTER_ID 7

static double bf16_value(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------ segments */

typedef struct {
    int32_t key;
    int32_t index;
} keyed_token;

static int by_key_then_index(const void *pa, const void *pb)
{
    const keyed_token *a = (const keyed_token *)pa, *b = (const keyed_token *)pb;
    if (a->key != b->key) return a->key < b->key ? -1 : 1;
    if (a->index != b->index) return a->index < b->index ? -1 : 1;
    return 0;
}

/*
 * ids[T]: -1 (base only) or a slot in [0, n_slots).
 * Outputs: order[T]; *n_base; *num_seg; seg_start[num_seg + 1] (offsets into
 * order; seg_start[0] = n_base, seg_start[num_seg] = T); seg_slot[num_seg]
 * (ascending). seg_start / seg_slot must hold min(T, n_slots) + 1 entries.
 */
int oracle_segments(const int32_t *ids, int64_t T, int32_t n_slots, int32_t *order,
                    int32_t *n_base, int32_t *num_seg, int32_t *seg_start, int32_t *seg_slot)
{
    if (T < 0 || n_slots < 0) return ORACLE_ERR_ARG;
    for (int64_t t = 0; t < T; ++t)
        if (ids[t] < -1 || ids[t] >= n_slots) return ORACLE_ERR_BAD_ADAPTER_ID;

    keyed_token *kt = (keyed_token *)malloc(sizeof(keyed_token) * (size_t)(T > 0 ? T : 1));
    if (!kt) return ORACLE_ERR_ARG;
    for (int64_t t = 0; t < T; ++t) {
        kt[t].key = ids[t];
        kt[t].index = (int32_t)t;
    }
    /* sorting by (id, token index) is the stable sort by id */
    qsort(kt, (size_t)T, sizeof(keyed_token), by_key_then_index);

    int32_t nb = 0, ns = 0;
    for (int64_t p = 0; p < T; ++p) {
        order[p] = kt[p].index;
        if (kt[p].key < 0) {
            ++nb;
        } else if (p == 0 || kt[p - 1].key != kt[p].key) {
            seg_start[ns] = (int32_t)p;
            seg_slot[ns] = kt[p].key;
            ++ns;
        }
    }
    seg_start[ns] = (int32_t)T;
    *n_base = nb;
    *num_seg = ns;
    free(kt);
    return ORACLE_OK;
}

/* ------------------------------------------------------------- lora linear */

/*
 * X[T x d_in], W[d_out x d_in] (nn.Linear layout), both bf16 bits, row-major.
 * A[i] -> bf16 [d_in x rank[i]] row-major, B[i] -> bf16 [rank[i] x d_out]
 * row-major, alpha[i]; A[i] == NULL marks an empty slot.
 * Y[T x d_out] double, row-major.
 * Returns ORACLE_ERR_BAD_ADAPTER_ID (writing nothing) if any id is neither -1
 * nor a loaded slot.
 */
int oracle_lora_linear(const uint16_t *X, const uint16_t *W, const int32_t *ids, int64_t T,
                       int64_t d_in, int64_t d_out, int32_t n_slots,
                       const uint16_t *const *A, const uint16_t *const *B,
                       const int32_t *rank, const double *alpha, double *Y)
{
    if (T < 0 || d_in <= 0 || d_out <= 0) return ORACLE_ERR_ARG;
    for (int64_t t = 0; t < T; ++t) {
        int32_t i = ids[t];
        if (i == -1) continue;
        if (i < -1 || i >= n_slots || A[i] == NULL || B[i] == NULL || rank[i] <= 0)
            return ORACLE_ERR_BAD_ADAPTER_ID;
    }

    int64_t max_r = 1;
    for (int32_t i = 0; i < n_slots; ++i)
        if (A[i] && rank[i] > max_r) max_r = rank[i];

#pragma omp parallel
    {
        double *u = (double *)malloc(sizeof(double) * (size_t)max_r);
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < T; ++t) {
            const uint16_t *x = X + t * d_in;
            const int32_t i = ids[t];

            /* low-rank intermediate u = X[t,:] A_i  (length r_i) */
            int64_t r = 0;
            double s = 0.0;
            if (i >= 0) {
                r = rank[i];
                s = alpha[i] / (double)r;
                for (int64_t j = 0; j < r; ++j) {
                    double acc = 0.0;
                    for (int64_t k = 0; k < d_in; ++k)
                        acc += bf16_value(x[k]) * bf16_value(A[i][k * r + j]);
                    u[j] = acc;
                }
            }

            for (int64_t n = 0; n < d_out; ++n) {
                /* base product  sum_k X[t,k] W[n,k] */
                const uint16_t *w = W + n * d_in;
                double base = 0.0;
                for (int64_t k = 0; k < d_in; ++k)
                    base += bf16_value(x[k]) * bf16_value(w[k]);

                /* low-rank branch  s * sum_j u[j] B_i[j,n] */
                double delta = 0.0;
                for (int64_t j = 0; j < r; ++j)
                    delta += u[j] * bf16_value(B[i][j * d_out + n]);

                Y[t * d_out + n] = base + s * delta;
            }
        }
        free(u);
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------ adapter chains */

/*
 * Several adapters on one token. Token t applies the adapters
 * list[off[t]] .. list[off[t+1] - 1] (an empty range: the base output only);
 * their low-rank branches add:
 *
 *   Y[t,n] = sum_k X[t,k] W[n,k]
 *          + sum over listed c of  s_c * sum_j ( sum_k X[t,k] A_c[k,j] ) B_c[j,n]
 *
 * Source: "LoRA-Land: 将大模型变成操作系统..." (blog), section 技术方案 item 3
 * (动态加载与组合: several adapters are combined like a pipeline and applied to
 * the kernel in order) and section 核心实现解析 / 3. 热插拔 API 与组合
 * (set_adaptive_chain). Applying the members' weight updates to one linear
 * layer one after another gives W + dW_a + dW_b, so at the layer the branches
 * add and their order does not change the result.
 * Same slot arrays as oracle_lora_linear; off has T + 1 entries, off[0] = 0,
 * non-decreasing. Returns ORACLE_ERR_BAD_ADAPTER_ID (writing nothing) if a
 * listed id is not a loaded slot, ORACLE_ERR_ARG for malformed offsets.
 */
int oracle_lora_linear_chains(const uint16_t *X, const uint16_t *W, const int32_t *off,
                              const int32_t *list, int64_t T, int64_t d_in, int64_t d_out,
                              int32_t n_slots, const uint16_t *const *A,
                              const uint16_t *const *B, const int32_t *rank,
                              const double *alpha, double *Y)
{
    if (T < 0 || d_in <= 0 || d_out <= 0 || off[0] != 0) return ORACLE_ERR_ARG;
    for (int64_t t = 0; t < T; ++t) {
        if (off[t + 1] < off[t]) return ORACLE_ERR_ARG;
        for (int32_t e = off[t]; e < off[t + 1]; ++e) {
            const int32_t c = list[e];
            if (c < 0 || c >= n_slots || A[c] == NULL || B[c] == NULL || rank[c] <= 0)
                return ORACLE_ERR_BAD_ADAPTER_ID;
        }
    }
    int64_t max_r = 1;
    for (int32_t c = 0; c < n_slots; ++c)
        if (A[c] && rank[c] > max_r) max_r = rank[c];

#pragma omp parallel
    {
        double *low = (double *)malloc(sizeof(double) * (size_t)max_r);
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < T; ++t) {
            const uint16_t *xt = X + t * d_in;
            double *yt = Y + t * d_out;
            /* the base row */
            for (int64_t n = 0; n < d_out; ++n) {
                double acc = 0.0;
                for (int64_t k = 0; k < d_in; ++k)
                    acc += bf16_value(xt[k]) * bf16_value(W[n * d_in + k]);
                yt[n] = acc;
            }
            /* each listed adapter's branch, added on */
            for (int32_t e = off[t]; e < off[t + 1]; ++e) {
                const int32_t c = list[e];
                const int64_t rc = rank[c];
                const double sc = alpha[c] / (double)rc;
                for (int64_t j = 0; j < rc; ++j) {
                    double acc = 0.0;
                    for (int64_t k = 0; k < d_in; ++k)
                        acc += bf16_value(xt[k]) * bf16_value(A[c][k * rc + j]);
                    low[j] = acc;
                }
                for (int64_t n = 0; n < d_out; ++n) {
                    double branch = 0.0;
                    for (int64_t j = 0; j < rc; ++j)
                        branch += low[j] * bf16_value(B[c][j * d_out + n]);
                    yt[n] += sc * branch;
                }
            }
        }
        free(low);
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------ quantised base (4-bit) */

/*
 * A base weight stored group-wise in 4 bits, dequantised to the activation type
 * (bfloat16) before the layer's product:
 *
 *   W[n,k] = bf16( s[g][n] * (q[n,k] - z[g][n]) ),   g = k / group
 *
 * Source: "多 LoRA 热插拔: 一模型服多租户" (vLLM tutorial), section 性能注意事项: the
 * base may be quantised to 4 bits (AWQ-INT4) while the adapters stay in bf16. The
 * pages give no format; the reading used: q an unsigned 4-bit code, two per byte
 * along k in the nn.Linear layout (Wq[n * d_in/2 + k/2], the even k in the low
 * nibble); per (group of `group` inputs, output row) one bf16 scale s and one
 * unsigned 4-bit zero point z (scales [d_in/group][d_out] as bf16 bits, zeros
 * [d_in/group][d_out] as bytes 0..15). The product s * (q - z) is exact in double
 * (an 8-bit significand times an integer of magnitude <= 15); it is rounded once to
 * bfloat16, to nearest with ties to even, as a dequantising kernel does before a
 * bf16 matrix product.
 * W receives d_out x d_in bf16 bit patterns. Returns ORACLE_ERR_ARG for a shape
 * that the groups do not divide or a zero point above 15.
 */
static uint16_t bf16_round_nearest_even(double v)
{
    float f = (float)v; /* exact: v has at most 12 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0x7FC0; /* NaN */
    /* round half to even on the 16 bits that are dropped */
    const uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

int oracle_dequant_q4(const uint8_t *Wq, const uint16_t *scales, const uint8_t *zeros,
                      int64_t d_out, int64_t d_in, int64_t group, uint16_t *W)
{
    if (d_out <= 0 || d_in <= 0 || group <= 0 || d_in % group != 0 || d_in % 2 != 0)
        return ORACLE_ERR_ARG;
    const int64_t groups = d_in / group;
    for (int64_t g = 0; g < groups; ++g)
        for (int64_t n = 0; n < d_out; ++n)
            if (zeros[g * d_out + n] > 15) return ORACLE_ERR_ARG;
    for (int64_t n = 0; n < d_out; ++n) {
        for (int64_t k = 0; k < d_in; ++k) {
            const uint8_t byte = Wq[n * (d_in / 2) + k / 2];
            const int q = (k % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
            const int64_t g = k / group;
            const int z = zeros[g * d_out + n];
            const double s = bf16_value(scales[g * d_out + n]);
            W[n * d_in + k] = bf16_round_nearest_even(s * (double)(q - z));
        }
    }
    return ORACLE_OK;
}
