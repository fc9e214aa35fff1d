/*
 * Oracle for batched paged-KV decode attention -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU restatement of what the decode path
 * computes, in IEEE double precision. Only the test suite, the smoke check and
 * the benchmark's CPU-baseline leg may load it. It shares no code, header,
 * table or helper with the CUDA library; the two meet only through the seeded
 * input bytes.
 *
 * Source of the definition: the "FlashInfer parity matrix" page, sections
 * "Admitted attention matrix" (paged batch decode: online softmax with an F32
 * softmax state; single decode split-K with partial workspace and a merge) and
 * "Domain coverage" (paged decode over NHD/HND pages; attention state merge).
 * Every attention row there is full (non-causal) attention over BF16 data with
 * head dimension 128; the oracle accepts any head dimension so that it can be
 * checked against brute force on tiny inputs.
 *
 * The pages print no formula. The oracle therefore writes out the textbook
 * definition of single-query attention over a gathered KV sequence:
 *     s_j   = sm_scale * sum_d q[d] * k_j[d]
 *     M     = max_j s_j,  Z = sum_j exp(s_j - M)
 *     out   = sum_j exp(s_j - M) * v_j / Z
 *     lse   = M + ln Z                     (natural logarithm)
 * with the readings listed in the design notes (consecutive query heads share
 * a KV head; CSR block tables with last_page_len in [1, page_size]).
 *
 * The causal prefill function follows the same page's row "Paged causal
 * prefill"; the RoPE and paged-append functions at the end follow its rows
 * "Standard RoPE" and "Fused RoPE plus paged append".
 *
 * Parity status: every function below is pinned by the not-gpu tests
 * (closed forms, invariants, brute force); none is "parity unpinned".
 */
#ifndef OXD_ORACLE_H
#define OXD_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Page layouts of the K and V pools (the pages name "NHD" and "HND"):
 *   NHD: element (page, t, h, d) at ((page*page_size + t)*num_kv_heads + h)*head_dim + d
 *   HND: element (page, h, t, d) at ((page*num_kv_heads + h)*page_size + t)*head_dim + d */
#define ORACLE_LAYOUT_NHD 0
#define ORACLE_LAYOUT_HND 1

/* Return codes. */
#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)   /* inconsistent shapes or block tables */
#define ORACLE_ENOMEM (-2)

/*
 * Paged decode attention in f64.
 *   q            bf16 bit patterns, [B][Hq][D]
 *   k, v         bf16 bit patterns, pools of num_pages pages in `layout`
 *   indptr       [B+1], indices [indptr[B]], last_page_len [B]
 *   heads        optional list of n_heads (b, hq) pairs, flattened as
 *                heads[2i] = b, heads[2i+1] = hq; NULL means every head,
 *                in which case out is [B][Hq][D] and lse is [B][Hq];
 *                otherwise out is [n_heads][D] and lse is [n_heads]
 *   nthreads     worker threads (<= 0: all online cores); the result does not
 *                depend on it
 * Returns ORACLE_OK, or ORACLE_EINVAL if a length is not positive, a
 * last_page_len is outside [1, page_size] or a page index is outside
 * [0, num_pages).
 */
int oracle_paged_decode_f64(int B, int Hq, int Hkv, int D, int page_size, int layout,
                            int64_t num_pages, const uint16_t* q, const uint16_t* k,
                            const uint16_t* v, const int32_t* indptr, const int32_t* indices,
                            const int32_t* last_page_len, double sm_scale,
                            const int32_t* heads, int n_heads, double* out, double* lse,
                            int nthreads);

/*
 * Attention state of one query head (b, hq) over the logical tokens
 * [tok_begin, tok_end) of request b (0 <= tok_begin <= tok_end <= L_b):
 * o = softmax-weighted mean of V over that range and lse = ln sum exp(s_j).
 * An empty range gives o = 0 and lse = -infinity.
 */
int oracle_partial_state_f64(int B, int Hq, int Hkv, int D, int page_size, int layout,
                             int64_t num_pages, const uint16_t* q, const uint16_t* k,
                             const uint16_t* v, const int32_t* indptr, const int32_t* indices,
                             const int32_t* last_page_len, double sm_scale, int b, int hq,
                             int64_t tok_begin, int64_t tok_end, double* o, double* lse);

/*
 * Merge of S attention states (v_i[D], s_i) of one head into one:
 *   M = max_i s_i, w_i = exp(s_i - M), out = sum w_i v_i / sum w_i,
 *   lse = M + ln sum w_i.
 * States with s_i = -infinity carry weight 0; if every s_i is -infinity the
 * result is out = 0, lse = -infinity.  v is [S][D].
 */
void oracle_merge_states_f64(int S, int D, const double* v, const double* s, double* out,
                             double* lse);

/*
 * Paged causal prefill attention in f64: the "FlashInfer parity matrix" page,
 * "Admitted attention matrix", row "Paged causal prefill" (BF16, D128, causal,
 * over the same NHD/HND pages and block tables as decode). Request b holds
 * L_b cached tokens and q_len_b = qo_indptr[b+1] - qo_indptr[b] query tokens,
 * which are its last q_len_b tokens (q_len_b <= L_b): query token i of
 * request b sits at position p = L_b - q_len_b + i and attends to cached
 * tokens 0 .. p:
 *     s_j = sm_scale * sum_d q[d] * k_j[d],   j = 0 .. p
 *     out = sum_j exp(s_j - M) v_j / Z,  lse = M + ln Z  (M = max s_j, Z = sum exp(s_j - M))
 * With q_len_b = 1 this is the decode above.
 *   q, out     [qo_indptr[B]][Hq][D]; lse [qo_indptr[B]][Hq]
 *   rows       optional list of n_rows (t, hq) pairs (t a global query token
 *              index), flattened; NULL = every (t, hq), in which case out and
 *              lse are full size, otherwise out is [n_rows][D], lse [n_rows]
 * Returns ORACLE_EINVAL for bad tables (as decode), a decreasing qo_indptr,
 * qo_indptr[0] != 0, or q_len_b > L_b.
 */
int oracle_paged_prefill_f64(int B, int Hq, int Hkv, int D, int page_size, int layout,
                             int64_t num_pages, const uint16_t* q, const uint16_t* k,
                             const uint16_t* v, const int32_t* qo_indptr, const int32_t* indptr,
                             const int32_t* indices, const int32_t* last_page_len,
                             double sm_scale, const int32_t* rows, int n_rows, double* out,
                             double* lse, int nthreads);

/* Logical token count of request b: (P_b - 1) * page_size + last_page_len[b]. */
int64_t oracle_kv_len(const int32_t* indptr, const int32_t* last_page_len, int page_size, int b);

/*
 * Standard rotary position embedding, split-half ("NeoX") pairing: the
 * "FlashInfer parity matrix" page, "Admitted attention matrix", row "Standard
 * RoPE" (D128 NeoX split-half with explicit int32 positions). For each of the
 * n rows x[D] (D even) at position pos[r], with h = D/2 and the frequencies
 * f_i = theta^(-2i/D), i < h:
 *     y_i     = x_i     cos(pos f_i) - x_{i+h} sin(pos f_i)
 *     y_{i+h} = x_{i+h} cos(pos f_i) + x_i     sin(pos f_i)
 * all in f64. `theta` is the frequency base (10000 in the standard variant).
 */
void oracle_rope_f64(int n, int D, const double* x, const int32_t* pos, double theta, double* y);

/* Round to the nearest bfloat16 (ties to even), returned as its bit pattern. */
uint16_t oracle_f64_to_bf16(double x);

/* Per-token outcome of oracle_rope_append. */
#define ORACLE_APPEND_WRITTEN 0
#define ORACLE_APPEND_SHARED_PAGE 1   /* target page's reference count is not one */
#define ORACLE_APPEND_BAD_POSITION 2  /* request outside [0, B) or position past its pages */
#define ORACLE_APPEND_BAD_PAGE 3      /* target page index outside [0, num_pages) */

/*
 * Fused RoPE and paged append: the "Admitted attention matrix" row "Fused
 * RoPE plus paged append" and the section "Paged KV ownership difference"
 * (decode may read shared pages; the append writes only to pages whose
 * reference count is one, and the pager makes a target private first).
 *
 * Token t (t < T) belongs to request b = token_request[t] at logical
 * position p = positions[t]; its KV rows go to page
 * indices[indptr[b] + p / page_size], slot p % page_size (the request's
 * block table already covers the position). For every KV head, the K row is
 * written as bf16(RoPE(k_t, p)) and the V row as v_t unchanged; for every
 * query head, q_out = bf16(RoPE(q_t, p)) (one rounding, ties to even).
 * A token whose target page has a reference count other than one, whose
 * request is outside [0, B), whose position is negative or past the
 * request's pages, or whose page index is outside [0, num_pages) writes
 * nothing to the pools (its q_out is still written); status[t] says which.
 *   q, q_out  bf16 bits [T][Hq][D];  k, v bf16 bits [T][Hkv][D]
 *   k_pages, v_pages  bf16 bits, pools in `layout`, updated in place
 * Returns the number of tokens not written, or ORACLE_EINVAL for bad shapes.
 */
int oracle_rope_append(int T, int B, int Hq, int Hkv, int D, int page_size, int layout,
                       int64_t num_pages, const uint16_t* q, const uint16_t* k,
                       const uint16_t* v, const int32_t* token_request, const int32_t* positions,
                       const int32_t* indptr, const int32_t* indices, const int32_t* refcount,
                       double theta, uint16_t* q_out, uint16_t* k_pages, uint16_t* v_pages,
                       int32_t* status);

#ifdef __cplusplus
}
#endif

#endif
