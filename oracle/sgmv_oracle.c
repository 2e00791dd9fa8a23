/*
 * sgmv_oracle.c -- the correctness oracle for segmented LoRA apply (SGMV), in plain C, fp64.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may load, link or call this file:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg use it.  It shares no
 * code, header, table or constant generator with the CUDA library; the two meet only through
 * the seeded inputs a test hands to both.
 *
 * What is computed, and where it comes from
 * -----------------------------------------
 * "Punica Guide: Multi-Tenant LoRA Serving with SGMV", section "The Heterogeneous Batching
 * Bottleneck: Why Standard Serving Stalls", the per-request equation
 *       y_i = x_i W0 + (alpha/r) x_i A_{k(i)} B_{k(i)},
 *   with A_k of shape d_in x r and B_k of shape r x d_out.  The caller supplies y already
 *   holding x_i W0 (the base output) and scale = alpha/r; the oracle adds the second term.
 * Same page, section "The SGMV Mathematical Formulation": tokens are grouped into contiguous
 *   segments [s_i, s_{i+1}), each bound to one adapter through a pointer array.  Segments are
 *   indexed 0..S-1 with S+1 offsets s_0..s_S (the page's "i in [1, N]" is read as the S
 *   segments between the S+1 offsets).
 * Same page, section "Step-by-Step Implementation: Multi-LoRA Batching Dispatcher in PyTorch":
 *   the reference semantics is a per-row loop x[i] @ A[id] @ B[id]; this file is that loop, in
 *   fp64, with the alpha/r factor of the equation above.
 *
 * Readings where the pages are silent (all stated again in the design notes):
 *   - y is accumulated into (+=), never overwritten: the equation's first term is the base
 *     output that already sits in y.
 *   - weights of adapter k are one contiguous block [L][h_in][r] (A) and [L][r][h_out] (B),
 *     row-major; layer_idx selects the [h_in][r] / [r][h_out] slice inside the block.
 *   - a segment whose adapter id is negative carries no adapter: its rows are left unchanged.
 *   - a segment with s_{i+1} <= s_i is empty.
 *
 * Every function here is pinned by the CPU tests (tests/test_oracle_pins.py) against closed
 * forms, library matmuls, brute force and invariants; none is "parity unpinned".
 */
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

/* Bits of the table check, as documented in the library header. */
#define ORACLE_BAD_ORDER    1  /* seg_starts decreases somewhere                     */
#define ORACLE_BAD_FIRST    2  /* seg_starts[0] < 0                                  */
#define ORACLE_BAD_LAST     4  /* seg_starts[S] > M                                  */
#define ORACLE_BAD_ADAPTER  8  /* adapter id >= num_adapters (negative = no adapter) */
#define ORACLE_BAD_A_PTR   16  /* a used adapter's A pointer is null or not 16-byte aligned */
#define ORACLE_BAD_B_PTR   32  /* the same for its B pointer                                */

/* v[t][c] = sum_j x[t][j] * A_k[layer][j][c]   for every row t of every segment.
 * "Shrink": the first factor of the equation, x_i A_k (h_in -> r).  v is [M][r]; rows outside
 * all segments are left as they are. */
int oracle_sgmv_shrink(double *v, const double *x, const double *const *A,
                       const int32_t *seg_starts, const int32_t *seg_adapter,
                       int32_t num_segments, int32_t layer_idx, int32_t h_in, int32_t r)
{
    for (int32_t i = 0; i < num_segments; ++i) {
        const int32_t k = seg_adapter[i];
        if (k < 0) continue;
        const double *Ak = A[k] + (size_t)layer_idx * (size_t)h_in * (size_t)r;
        for (int32_t t = seg_starts[i]; t < seg_starts[i + 1]; ++t) {
            const double *xt = x + (size_t)t * (size_t)h_in;
            double *vt = v + (size_t)t * (size_t)r;
            for (int32_t c = 0; c < r; ++c) {
                double s = 0.0;
                for (int32_t j = 0; j < h_in; ++j)
                    s += xt[j] * Ak[(size_t)j * (size_t)r + (size_t)c];
                vt[c] = s;
            }
        }
    }
    return 0;
}

/* y[t][n] += scale * sum_c v[t][c] * B_k[layer][c][n]   for every row t of every segment.
 * "Expand": the second factor, (x_i A_k) B_k (r -> h_out), times alpha/r, added into y. */
int oracle_sgmv_expand(double *y, const double *v, const double *const *B,
                       const int32_t *seg_starts, const int32_t *seg_adapter,
                       int32_t num_segments, int32_t layer_idx, int32_t r, int32_t h_out,
                       double scale)
{
    for (int32_t i = 0; i < num_segments; ++i) {
        const int32_t k = seg_adapter[i];
        if (k < 0) continue;
        const double *Bk = B[k] + (size_t)layer_idx * (size_t)r * (size_t)h_out;
        for (int32_t t = seg_starts[i]; t < seg_starts[i + 1]; ++t) {
            const double *vt = v + (size_t)t * (size_t)r;
            double *yt = y + (size_t)t * (size_t)h_out;
            for (int32_t n = 0; n < h_out; ++n) {
                double s = 0.0;
                for (int32_t c = 0; c < r; ++c)
                    s += vt[c] * Bk[(size_t)c * (size_t)h_out + (size_t)n];
                yt[n] += scale * s;
            }
        }
    }
    return 0;
}

/* y[t] += scale * (x[t] A_k) B_k   -- the whole LoRA term, one token at a time, one segment
 * after another (the per-row loop of the dispatcher listing, with the alpha/r factor). */
int oracle_lora_apply(double *y, const double *x, const double *const *A,
                      const double *const *B, const int32_t *seg_starts,
                      const int32_t *seg_adapter, int32_t num_segments, int32_t layer_idx,
                      int32_t h_in, int32_t h_out, int32_t r, double scale)
{
    double *v = (double *)malloc(sizeof(double) * (size_t)(r > 0 ? r : 1));
    if (!v) return -1;
    for (int32_t i = 0; i < num_segments; ++i) {
        const int32_t k = seg_adapter[i];
        if (k < 0) continue;
        const double *Ak = A[k] + (size_t)layer_idx * (size_t)h_in * (size_t)r;
        const double *Bk = B[k] + (size_t)layer_idx * (size_t)r * (size_t)h_out;
        for (int32_t t = seg_starts[i]; t < seg_starts[i + 1]; ++t) {
            const double *xt = x + (size_t)t * (size_t)h_in;
            double *yt = y + (size_t)t * (size_t)h_out;
            for (int32_t c = 0; c < r; ++c) {
                double s = 0.0;
                for (int32_t j = 0; j < h_in; ++j)
                    s += xt[j] * Ak[(size_t)j * (size_t)r + (size_t)c];
                v[c] = s;
            }
            for (int32_t n = 0; n < h_out; ++n) {
                double s = 0.0;
                for (int32_t c = 0; c < r; ++c)
                    s += v[c] * Bk[(size_t)c * (size_t)h_out + (size_t)n];
                yt[n] += scale * s;
            }
        }
    }
    free(v);
    return 0;
}

/* Checks a segment table the way the library's validation entry point documents it.
 * Returns an OR of the ORACLE_BAD_* bits (0 = valid). */
int32_t oracle_validate(const int32_t *seg_starts, const int32_t *seg_adapter,
                        int32_t num_segments, int32_t num_adapters, int32_t M)
{
    int32_t bits = 0;
    if (num_segments < 0) return ORACLE_BAD_ORDER;
    if (seg_starts[0] < 0) bits |= ORACLE_BAD_FIRST;
    if (seg_starts[num_segments] > M) bits |= ORACLE_BAD_LAST;
    for (int32_t i = 0; i < num_segments; ++i) {
        if (seg_starts[i + 1] < seg_starts[i]) bits |= ORACLE_BAD_ORDER;
        if (seg_adapter[i] >= num_adapters) bits |= ORACLE_BAD_ADAPTER;
    }
    return bits;
}

/* Checks the per-adapter weight addresses that the segment table will dereference ("Punica
 * Guide: Multi-Tenant LoRA Serving with SGMV", section "Core Innovation 1", figure "SGMV Kernel
 * Memory Layout & Execution Grid": a pointer array to each adapter's contiguous weights).
 * A_addr / B_addr hold the addresses as integers (either may be NULL: not checked).  Only
 * adapters of non-empty segments with 0 <= id < num_adapters are looked at.  Returns an OR of
 * ORACLE_BAD_A_PTR / ORACLE_BAD_B_PTR (0 = valid). */
int32_t oracle_validate_pointers(const uint64_t *A_addr, const uint64_t *B_addr,
                                 const int32_t *seg_starts, const int32_t *seg_adapter,
                                 int32_t num_segments, int32_t num_adapters)
{
    int32_t bits = 0;
    for (int32_t i = 0; i < num_segments; ++i) {
        const int32_t k = seg_adapter[i];
        if (k < 0 || k >= num_adapters || seg_starts[i + 1] <= seg_starts[i]) continue;
        if (A_addr && (A_addr[k] == 0 || A_addr[k] % 16 != 0)) bits |= ORACLE_BAD_A_PTR;
        if (B_addr && (B_addr[k] == 0 || B_addr[k] % 16 != 0)) bits |= ORACLE_BAD_B_PTR;
    }
    return bits;
}

/* The adapter grouping that a plan of the table holds ("Punica Guide: Multi-Tenant LoRA Serving
 * with SGMV", section "Hardware-Level Optimizations in SGMV": segment descriptors pre-sorted so
 * that each adapter's weights are streamed once; section "Mathematical Modeling: Throughput
 * Scaling and Kernel Launch Bounds", part 2: the work list is built once and reused by every
 * layer's launches).  Groups are the distinct adapter ids >= 0 of non-empty segments, in the
 * order of their first segment; a group's rows are its segments' rows, segment after segment,
 * each segment's rows in increasing order.  Writes g_starts[G+1] (row offsets of the groups in
 * rows[]), g_adapter[G] and rows[] (token indices); returns G, or -1 when more than max_rows
 * rows would be listed. */
int32_t oracle_plan(const int32_t *seg_starts, const int32_t *seg_adapter, int32_t num_segments,
                    int32_t max_rows, int32_t *g_starts, int32_t *g_adapter, int32_t *rows)
{
    int32_t G = 0, n = 0;
    for (int32_t i = 0; i < num_segments; ++i) {
        const int32_t k = seg_adapter[i];
        if (k < 0 || seg_starts[i + 1] <= seg_starts[i]) continue;
        int32_t seen = 0;
        for (int32_t g = 0; g < G; ++g)
            if (g_adapter[g] == k) seen = 1;
        if (seen) continue;
        /* first segment of adapter k: collect every segment of k from here on, in order */
        g_adapter[G] = k;
        g_starts[G] = n;
        for (int32_t j = i; j < num_segments; ++j) {
            if (seg_adapter[j] != k) continue;
            for (int32_t t = seg_starts[j]; t < seg_starts[j + 1]; ++t) {
                if (n >= max_rows) return -1;
                rows[n++] = t;
            }
        }
        ++G;
    }
    g_starts[G] = n;
    return G;
}

/* y[t] += scale_k * (x[t] A_k) B_k with a rank and a scale of its own for every adapter
 * ("Punica Guide: Multi-Tenant LoRA Serving with SGMV", section "The Heterogeneous Batching
 * Bottleneck", the y_i equation with alpha/r taken per adapter, A_k of shape d_in x r_k and B_k
 * of shape r_k x d_out; section "Operational Checklist", rank standardisation: batches whose
 * adapters differ in rank).  A[k] is adapter k's block [L][h_in][rank[k]], B[k] its block
 * [L][rank[k]][h_out]; scale[k] multiplies its term.  Same per-row loop as oracle_lora_apply. */
int oracle_lora_apply_ranked(double *y, const double *x, const double *const *A,
                             const double *const *B, const int32_t *rank, const double *scale,
                             const int32_t *seg_starts, const int32_t *seg_adapter,
                             int32_t num_segments, int32_t layer_idx, int32_t h_in,
                             int32_t h_out)
{
    int32_t r_max = 1;
    for (int32_t i = 0; i < num_segments; ++i)
        if (seg_adapter[i] >= 0 && rank[seg_adapter[i]] > r_max) r_max = rank[seg_adapter[i]];
    double *v = (double *)malloc(sizeof(double) * (size_t)r_max);
    if (!v) return -1;
    for (int32_t i = 0; i < num_segments; ++i) {
        const int32_t k = seg_adapter[i];
        if (k < 0) continue;
        const int32_t r = rank[k];
        const double *Ak = A[k] + (size_t)layer_idx * (size_t)h_in * (size_t)r;
        const double *Bk = B[k] + (size_t)layer_idx * (size_t)r * (size_t)h_out;
        for (int32_t t = seg_starts[i]; t < seg_starts[i + 1]; ++t) {
            const double *xt = x + (size_t)t * (size_t)h_in;
            double *yt = y + (size_t)t * (size_t)h_out;
            for (int32_t c = 0; c < r; ++c) {
                double s = 0.0;
                for (int32_t j = 0; j < h_in; ++j)
                    s += xt[j] * Ak[(size_t)j * (size_t)r + (size_t)c];
                v[c] = s;
            }
            for (int32_t n = 0; n < h_out; ++n) {
                double s = 0.0;
                for (int32_t c = 0; c < r; ++c)
                    s += v[c] * Bk[(size_t)c * (size_t)h_out + (size_t)n];
                yt[n] += scale[k] * s;
            }
        }
    }
    free(v);
    return 0;
}

/* y[t] = x[t] W0 + scale * (x[t] A_k) B_k -- both terms of the per-request equation
 * ("Punica Guide: Multi-Tenant LoRA Serving with SGMV", section "The Heterogeneous Batching
 * Bottleneck", y_i = x_i W0 + (alpha/r) x_i A B, and the figure of the same section in which
 * the base GEMM feeds the fused SGMV kernel; section "Step-by-Step Implementation", the
 * dispatcher's base output plus its delta).  The base weight is stored as a linear layer
 * keeps it, one row per output feature: W0 is [h_out][h_in] row-major, so the equation's
 * x_i W0 is sum_j x[t][j] * W0[n][j].  y is written, not accumulated: every row t < M gets
 * its base projection, and the rows of segments with an adapter (id >= 0) get the LoRA term
 * on top (by oracle_lora_apply, the same per-row loop). */
int oracle_base_lora(double *y, const double *x, const double *W0, const double *const *A,
                     const double *const *B, const int32_t *seg_starts,
                     const int32_t *seg_adapter, int32_t num_segments, int32_t M,
                     int32_t layer_idx, int32_t h_in, int32_t h_out, int32_t r, double scale)
{
    for (int32_t t = 0; t < M; ++t) {
        const double *xt = x + (size_t)t * (size_t)h_in;
        double *yt = y + (size_t)t * (size_t)h_out;
        for (int32_t n = 0; n < h_out; ++n) {
            const double *wn = W0 + (size_t)n * (size_t)h_in;
            double s = 0.0;
            for (int32_t j = 0; j < h_in; ++j)
                s += xt[j] * wn[j];
            yt[n] = s;
        }
    }
    return oracle_lora_apply(y, x, A, B, seg_starts, seg_adapter, num_segments, layer_idx, h_in,
                             h_out, r, scale);
}
