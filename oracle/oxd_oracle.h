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

/* Logical token count of request b: (P_b - 1) * page_size + last_page_len[b]. */
int64_t oracle_kv_len(const int32_t* indptr, const int32_t* last_page_len, int page_size, int b);

#ifdef __cplusplus
}
#endif

#endif
