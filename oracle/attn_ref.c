/*
 * attn_ref.c -- fp64 CPU oracle for paged, relative-bias, grouped-query attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously-correct
 * definition that the CUDA library is checked against.  Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg may load it.  It shares no code,
 * header or constant with the CUDA path.
 *
 * What it computes (one output row per packed query row t and query head h):
 *
 *   sequence b owns packed rows [cu_q[b], cu_q[b+1]); n_b = cu_q[b+1] - cu_q[b]
 *   new tokens are the LAST n_b positions of a KV history of length L_b = seq_lens[b],
 *   so row i of sequence b sits at absolute position  p = L_b - n_b + i
 *   g = h / (Hq / Hkv)                                   -- GQA head map
 *   visible keys:  0 <= k <= p  and, when window > 0,  p - k <= window - 1
 *   page of key k: block_table[b][k / P], slot k % P      -- positional page table
 *   s_k = sm_scale * sum_d q[t,h,d] K[page,g,slot,d]  +  rel[t, h, min(p - k, E - 1)]
 *   out[t,h,:] = sum_k softmax(s)_k V[page,g,slot,:]
 *
 * Sources (pages of the web capture this project is built from):
 *  - "Support Inkling-NVFP4 model" (TensorRT-LLM PR #17062), section "Architecture":
 *    no RoPE; a learned relative-position bias per (query token, head, relative
 *    distance) is ADDED BEFORE the softmax; local layers use a 512-key sliding window
 *    (16 KV heads), global layers are full causal (8 KV heads).
 *  - same page, section "Implementation", row attention_backend/inkling_triton.py:
 *    paged prefill + decode kernels that apply the bias as a score modifier.
 *  - same page, review of _build_rel_logits: the bias tensor is [T, heads, rel_extent]
 *    in fp32.
 *  - "Inkling attn backend cleanup fake registry" (TensorRT-LLM PR #17860), commit on
 *    GQA input checks: query head -> KV head is cur_head // (num_heads // num_kv_heads),
 *    and a non-divisible pair is an error.
 *  - same page, commit that moves attention into the backend: the per-layer scalars
 *    are sm_scale, rel_extent and window_left; a global layer has window_left = -1.
 *  - same page, commits on borrowing the base page table: the kernels address a page as
 *    k_pos // page_size through a positional table, and k_pos < seq_len bounds every
 *    access, so table entries past a request's own blocks are never read.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - window W keeps the W keys at distances 0..W-1 (self included); W <= 0 = no window;
 *  - distances >= E-1 all use bucket E-1 (clamp);
 *  - the bias is not multiplied by sm_scale;
 *  - a sequence with L_b == 0 produces zeros;
 *  - masked keys are simply absent from the sum (no finite "-inf" stand-in is needed
 *    in exact arithmetic).
 *
 * Error behaviour: returns 0 on success, a negative code when the inputs break the
 * contract (bad shapes, n_b > L_b, a page id out of range for a visible key).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the high half of an IEEE binary32; widening it is exact. */
static double bf16_to_f64(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Find the sequence that owns packed query row t (cu_q is non-decreasing). */
static int owner_of_row(const int32_t* cu_q, int num_seqs, int64_t t) {
    int lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if ((int64_t)cu_q[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

/*
 * Compute n_rows output rows.  Row r is (packed query row row_t[r], query head row_h[r]);
 * its D values go to out[r*D .. r*D+D-1].  Passing every (t, h) pair gives the full
 * output; passing a sample gives those rows only.
 *
 * q:           [total_q, Hq, D] bf16 bits
 * k_cache/v_cache: [num_pages, Hkv, P, D] bf16 bits
 * block_table: [num_seqs, max_pages] int32
 * rel:         [total_q, Hq, E] fp32
 * q_rows, rel_rows: optional (may be NULL).  When given, the query vector and bias row
 *              of output row r are q_rows[r*D ..] and rel_rows[r*E ..] instead of
 *              q[t, h, :] and rel[t, h, :] (lets a caller pass only the sampled rows of a
 *              problem too large to copy whole; q / rel are then unused).
 */
int oracle_attention_rows(
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int page_size, int max_pages, int num_pages, int rel_extent, int window,
    double sm_scale,
    const int32_t* cu_q, const int32_t* seq_lens,
    const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
    const int32_t* block_table, const float* rel,
    int64_t n_rows, const int32_t* row_t, const int32_t* row_h,
    const uint16_t* q_rows, const float* rel_rows,
    double* out)
{
    if (num_seqs < 1 || num_q_heads < 1 || num_kv_heads < 1 || head_dim < 1) return -1;
    if (num_q_heads % num_kv_heads != 0) return -1;
    if (page_size < 1 || max_pages < 0 || num_pages < 0 || rel_extent < 1) return -1;
    const int group = num_q_heads / num_kv_heads;
    const int64_t total_q = cu_q[num_seqs];
    int status = 0;

#pragma omp parallel
    {
        double* s = NULL;      /* scores of the visible keys of one row */
        int64_t cap = 0;
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < n_rows; ++r) {
            double* o = out + r * head_dim;
            for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
            const int64_t t = row_t[r];
            const int h = row_h[r];
            if (t < 0 || t >= total_q || h < 0 || h >= num_q_heads) {
#pragma omp atomic write
                status = -2;
                continue;
            }
            const int b = owner_of_row(cu_q, num_seqs, t);
            const int64_t n_b = (int64_t)cu_q[b + 1] - cu_q[b];
            const int64_t L = seq_lens[b];
            if (L == 0) continue;                       /* padding row: zeros */
            if (n_b > L || L > (int64_t)max_pages * page_size) {
#pragma omp atomic write
                status = -3;
                continue;
            }
            const int64_t p = L - n_b + (t - cu_q[b]);  /* absolute position */
            const int g = h / group;                    /* GQA map */
            int64_t lo = 0;
            if (window > 0 && p - (window - 1) > 0) lo = p - (window - 1);
            const int64_t n_vis = p - lo + 1;
            if (n_vis > cap) {
                free(s);
                cap = n_vis;
                s = (double*)malloc((size_t)cap * sizeof(double));
            }
            const uint16_t* qrow = q_rows ? q_rows + r * (int64_t)head_dim
                                          : q + (t * num_q_heads + h) * (int64_t)head_dim;
            const float* brow = rel_rows ? rel_rows + r * (int64_t)rel_extent
                                         : rel + (t * num_q_heads + h) * (int64_t)rel_extent;
            int bad = 0;
            double m = -INFINITY;
            for (int64_t k = lo; k <= p; ++k) {
                const int32_t page = block_table[(int64_t)b * max_pages + k / page_size];
                if (page < 0 || page >= num_pages) { bad = 1; break; }
                const int64_t slot = k % page_size;
                const uint16_t* krow =
                    k_cache + (((int64_t)page * num_kv_heads + g) * page_size + slot) * head_dim;
                double dot = 0.0;
                for (int d = 0; d < head_dim; ++d) dot += bf16_to_f64(qrow[d]) * bf16_to_f64(krow[d]);
                int64_t dist = p - k;
                if (dist > rel_extent - 1) dist = rel_extent - 1;
                const double sk = sm_scale * dot + (double)brow[dist];
                s[k - lo] = sk;
                if (sk > m) m = sk;
            }
            if (bad) {
#pragma omp atomic write
                status = -4;
                continue;
            }
            double denom = 0.0;
            for (int64_t k = lo; k <= p; ++k) {
                const double w = exp(s[k - lo] - m);
                denom += w;
                const int32_t page = block_table[(int64_t)b * max_pages + k / page_size];
                const int64_t slot = k % page_size;
                const uint16_t* vrow =
                    v_cache + (((int64_t)page * num_kv_heads + g) * page_size + slot) * head_dim;
                for (int d = 0; d < head_dim; ++d) o[d] += w * bf16_to_f64(vrow[d]);
            }
            for (int d = 0; d < head_dim; ++d) o[d] /= denom;
        }
        free(s);
    }
    return status;
}
