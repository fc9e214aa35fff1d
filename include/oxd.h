/*
 * oxd -- batched paged-KV decode attention for NVIDIA GB300 (sm_103a).
 *
 * One BF16 query token per request attends, with full softmax attention, over
 * that request's KV cache, which lives in fixed-size pages of a shared K pool
 * and V pool and is addressed through CSR block tables
 * (indptr / indices / last_page_len). MHA, GQA and MQA head groupings; NHD or
 * HND page layout; head dimension 128.
 *
 * What the operation is: the "FlashInfer parity matrix" page, section
 * "Admitted attention matrix", row "Paged batch decode" (MHA, MQA, GQA, mixed
 * lengths, page order, read-only page reuse), with the softmax state kept in
 * F32 as every attention row there fixes; "Domain coverage" names the NHD and
 * HND paged layouts; the "Single decode split-K" row gives split partitions with
 * an F32 partial workspace followed by a merge; "Attention state and cascade"
 * names the state merge.
 *
 * How it is driven: the "Oxide Infer" README, section "One execution model"
 * (spec -> plan -> operands -> command scope -> completion; planning fixes the
 * algorithm, workspace and launch configuration and enqueue never tunes or
 * falls back) and section "Providers" (caller-selected stream, checked span,
 * alignment, alias and capacity rules, explicit workspace requirements,
 * completion-owned resource leases, typed device-status failures).
 *
 * Conventions for every entry point:
 *  - Returns an oxd_status. On any error nothing has been enqueued and no
 *    caller memory has been written.
 *  - "device" pointers are CUDA device (or managed) addresses on the plan's
 *    device; "host" pointers are ordinary host memory read during the call.
 *  - The caller owns every buffer and the stream. The library allocates no
 *    device memory and never synchronises a stream, except
 *    oxd_read_device_status, which says so.
 *  - Streams are passed as void* and are cudaStream_t values (NULL = the
 *    legacy default stream).
 *
 * Numerics: logits, the running maximum, the softmax denominator and the
 * output accumulator are F32; QK^T and PV products run on tensor cores for
 * grouped heads (Hq/Hkv >= 3) with BF16 operands (the softmax weights P are
 * rounded to BF16 before the PV product) and on CUDA cores for Hq/Hkv <= 2.
 * out is rounded once to BF16 (nearest even). lse is the natural logarithm of
 * sum_j exp(sm_scale * q.k_j). Results are deterministic: the same plan and
 * inputs give bitwise identical out and lse (no floating-point atomics).
 */
#ifndef OXD_H
#define OXD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    OXD_OK = 0,
    OXD_ERR_INVALID_ARGUMENT = 1,   /* bad shape, NULL pointer, bad block table */
    OXD_ERR_UNSUPPORTED = 2,        /* valid request outside the implemented contract */
    OXD_ERR_ALIGNMENT = 3,          /* a pointer misses its required alignment */
    OXD_ERR_ALIAS = 4,              /* an output overlaps an input or another output */
    OXD_ERR_WORKSPACE_TOO_SMALL = 5,
    OXD_ERR_PLAN_MISMATCH = 6,      /* plan used with another device, or a destroyed plan */
    OXD_ERR_CUDA = 7,               /* a CUDA runtime call failed (launch, copy, query) */
    OXD_ERR_DEVICE_STATUS = 8,      /* the kernels reported an error; see the code */
    OXD_ERR_NO_MEMORY = 9           /* host allocation failed while planning */
} oxd_status;

typedef enum {
    /* page = [page_size][num_kv_heads][head_dim]; element (p, t, h, d) at
     * ((p*page_size + t)*num_kv_heads + h)*head_dim + d */
    OXD_LAYOUT_NHD = 0,
    /* page = [num_kv_heads][page_size][head_dim]; element (p, h, t, d) at
     * ((p*num_kv_heads + h)*page_size + t)*head_dim + d */
    OXD_LAYOUT_HND = 1
} oxd_kv_layout;

/* Codes the kernels write into the workspace status word (first error wins). */
#define OXD_DEVICE_OK 0
#define OXD_DEVICE_BAD_PAGE 1       /* a listed page index is outside [0, num_pages) */
#define OXD_DEVICE_PLAN_MISMATCH 2  /* device indptr/last_page_len differ from the plan's */
#define OXD_DEVICE_WAIT_TIMEOUT 3   /* an internal pipeline wait gave up (about 1 s) */
#define OXD_DEVICE_SHARED_PAGE 4    /* an append targeted a page whose reference count is not 1 */
#define OXD_DEVICE_BAD_POSITION 5   /* an append's request or position lies outside its table */

typedef struct oxd_plan_s* oxd_plan; /* opaque, host-owned, immutable after planning */

typedef struct {
    int32_t batch;          /* B >= 1 requests, one query token each */
    int32_t num_qo_heads;   /* Hq >= 1 */
    int32_t num_kv_heads;   /* Hkv >= 1, Hq % Hkv == 0, G = Hq/Hkv <= 32 */
    int32_t head_dim;       /* D; must be 128 */
    int32_t page_size;      /* ps in {8, 16, 32, 64} tokens */
    int32_t layout;         /* oxd_kv_layout */
    int64_t num_pages;      /* pages in each of the K and V pools; 1 <= num_pages < 2^31 */
    int32_t max_splits;     /* 0 = planner's choice; 1 = never split; n = at most n per request */
    int32_t force_splits;   /* 0 = off; n > 0: split every request into min(n, P_b) chunks */
    int32_t num_sms;        /* 0 = query the device; > 0 = plan for that many SMs */
    int32_t tensor_path;    /* groups of 17..32 query heads: 0 = tcgen05 (TMEM accumulators,
                               one CTA per piece), 1 = mma.sync (pairs of 16-row CTAs);
                               other groups ignore it */
    /* Cascade ("Attention state and cascade"; "Paged KV ownership difference":
     * decode may read shared pages): 0, 0 = off. Otherwise requests
     * [g*share_group, (g+1)*share_group) share the pages of their first
     * shared_prefix_tokens cached tokens (the caller guarantees that their first
     * shared_prefix_tokens / page_size block-table entries are the same pages).
     * The plan then attends each group's requests to that prefix once (on the
     * tensor cores, every query row of the group against each prefix page read
     * once), decodes the rest of every request, and merges the two states;
     * results equal the plain decode's within rounding. A request whose L_b is
     * not above shared_prefix_tokens, or that is alone in its group, is decoded
     * whole. */
    int32_t shared_prefix_tokens; /* 0, or a positive multiple of page_size */
    int32_t share_group;          /* 0 (with no prefix), or >= 2 consecutive requests */
    /* 1: launch a run's first kernel as a programmatic dependent of the kernel
     * before it on the stream (e.g. oxd_rope_append writing this step's q and
     * K/V rows): its CTAs are scheduled while that kernel finishes, and they
     * wait for it to complete (griddepcontrol.wait) before they read or write
     * any memory, so the results are those of a plain launch. The kernel
     * before it gains from triggering its dependents early
     * (griddepcontrol.launch_dependents), as oxd_rope_append does; a copy or
     * event between the two launches makes it a plain launch. Not used while
     * timing events are set. 0: plain launches. */
    int32_t pdl;
    /* How long one pipeline wait inside the kernels may last before the run
     * gives up ("Providers": typed device-status failures): 0 = about one
     * second; n > 0 = n nanoseconds. A run whose wait runs out stops its
     * CTA, records OXD_DEVICE_WAIT_TIMEOUT and returns; before the CTA
     * leaves it still waits (up to about one second, whatever this limit)
     * for the copies and tensor-core operations it has already issued.
     * The outputs of such a run are unspecified; the next run is unaffected.
     * A limit of a few nanoseconds makes most runs give up (a test of that
     * path). */
    int64_t wait_timeout_ns;
} oxd_paged_decode_desc;

typedef struct {
    int32_t num_work_items;     /* (request, page-range) chunks; work units = this x Hkv */
    int32_t num_split_requests; /* requests whose chunks need a merge */
    int32_t max_chunks;         /* most chunks any request got */
    int32_t chunk_pages;        /* planner's chunk length in pages */
    int32_t num_slots;          /* partial-state slots in the workspace */
    int32_t kernel_variant;     /* 0/1: CUDA-core G=1/G=2; 2,3,4: tensor-core G<=8, <=16, <=32 */
    int32_t grid_ctas;          /* persistent decode CTAs launched per run */
    int32_t ctas_per_sm;        /* resident decode CTAs per SM assumed by the planner */
    int32_t num_sms;
    int32_t launches_per_run;   /* kernels one run enqueues: decode, plus merge if split */
    int64_t workspace_bytes;
    int64_t upload_bytes;       /* host->device bytes one run copies (0: work list fits the
                                   kernel parameter buffer) */
    int64_t total_kv_tokens;    /* sum_b L_b */
    int32_t cascade_units;      /* prefix tiles (group chunk x KV head) of a cascade plan, else 0 */
    int32_t cascade_requests;   /* requests decoded as prefix + suffix */
    int64_t shared_kv_tokens;   /* cached tokens read once per group instead of once per request
                                   (sum over cascade requests of shared_prefix_tokens, minus
                                   one prefix per tile), 0 without cascade */
    int32_t cluster_size;       /* > 0: every (request, KV head) stream is cut into this many
                                   pieces run by one thread-block cluster, whose first CTA
                                   merges them (one launch per run); 0: no cluster merge */
    int32_t reserved;
} oxd_plan_info;

/*
 * Plan one batch of decode ("One execution model": the plan fixes the
 * algorithm, the split of each request's pages into chunks, the launch shape
 * and the workspace size; a run never re-plans).
 *
 *   desc               shapes and options (host)
 *   indptr_host        [B+1] int32, host: request b owns index entries
 *                      [indptr[b], indptr[b+1]); at least one page each;
 *                      non-decreasing, indptr[0] >= 0
 *   last_page_len_host [B] int32, host: tokens used in request b's last page,
 *                      in [1, page_size]; L_b = (P_b - 1)*page_size + last
 *   device             CUDA device ordinal the plan will run on (ignored when
 *                      desc->num_sms > 0; then planning makes no device query)
 *   plan_out           receives the plan; destroy with oxd_plan_destroy
 *   workspace_bytes_out receives the device workspace size run needs
 *
 * How the work is cut is the plan's choice (reported by oxd_plan_get_info):
 * the page streams of all (request, KV head) pairs are laid end to end and
 * cut into one share per resident CTA, streams cut in two or more being
 * merged by a second kernel; or, for a small batch of groups of up to 8
 * heads (every stream at least C >= 2 pages, C <= 8, and B * Hkv * C CTAs
 * resident at once), each stream is cut into C pieces run by one
 * thread-block cluster whose first CTA merges them: one launch.
 * A run passes the work list to the kernels in their parameter buffers; a
 * list too long for them is kept page-locked by the plan and copied to the
 * workspace asynchronously by each run, so the plan must outlive every run
 * that used it until that run's stream work has completed.
 * Errors: OXD_ERR_INVALID_ARGUMENT (NULL pointer, non-positive sizes,
 * Hq % Hkv != 0, empty request, last_page_len outside [1, page_size], a
 * shared_prefix_tokens that is negative or not a multiple of page_size, a
 * share_group below 2 with a prefix, or a share_group without one),
 * OXD_ERR_UNSUPPORTED (head_dim != 128, page_size not in
 * {8,16,32,64}, G > 32), OXD_ERR_CUDA (device query failed),
 * OXD_ERR_NO_MEMORY.
 */
oxd_status oxd_paged_decode_plan(const oxd_paged_decode_desc* desc, const int32_t* indptr_host,
                                 const int32_t* last_page_len_host, int device,
                                 oxd_plan* plan_out, size_t* workspace_bytes_out);

/*
 * Enqueue one decode step on `stream` ("Paged batch decode" row of
 * "Admitted attention matrix"):
 *   out[b, hq, :] = sum_j softmax_j(sm_scale * q[b, hq, :] . k_j) v_j
 *   lse[b, hq]    = ln sum_j exp(sm_scale * q[b, hq, :] . k_j)
 * over the L_b tokens of request b, taken from pages
 * indices[indptr[b] .. indptr[b+1]) in order, KV head h = hq / (Hq/Hkv).
 *
 *   q             device bf16 [B][Hq][128], 16-byte aligned
 *   k_pages       device bf16 pool of num_pages pages in the plan's layout,
 *   v_pages       16-byte aligned; read only (pages may be listed by many
 *                 requests -- read-only page reuse)
 *   indptr        device int32 [B+1], same values as the plan's host copy
 *   indices       device int32 [indptr[B]], physical page of each logical page
 *   last_page_len device int32 [B], same values as the plan's host copy
 *   sm_scale      finite logit scale (no implicit 1/sqrt(D))
 *   out           device bf16 [B][Hq][128], 16-byte aligned
 *   lse           device f32 [B][Hq], 4-byte aligned, or NULL
 *   workspace     device scratch of at least the planned size, 256-byte
 *                 aligned, any contents (nothing needs zeroing) unless it is
 *                 bound to this plan (oxd_plan_bind_workspace); holds the
 *                 device status word, the split partial states and, when
 *                 bound or when the work list is too long for the kernel's
 *                 parameter buffer, the work list; must not be shared by runs
 *                 that can overlap on the GPU
 *   stream        cudaStream_t
 *
 * Host-side errors (nothing enqueued): OXD_ERR_INVALID_ARGUMENT,
 * OXD_ERR_ALIGNMENT, OXD_ERR_ALIAS (out, lse and workspace must not overlap
 * each other or any input), OXD_ERR_WORKSPACE_TOO_SMALL,
 * OXD_ERR_PLAN_MISMATCH (destroyed plan, or the calling thread's current
 * device differs from the plan's), OXD_ERR_CUDA (copy or launch failed).
 * Device-side errors (an out-of-range page index, device block tables that
 * differ from the plan's) do not fault: the kernels record a code in the
 * workspace status word, read with oxd_read_device_status; out/lse of the
 * affected heads are then unspecified (finite for a bad page: the kernel
 * reads page 0 in its place, so no access leaves the pools).
 */
oxd_status oxd_paged_decode_run(oxd_plan plan, const void* q, const void* k_pages,
                                const void* v_pages, const int32_t* indptr,
                                const int32_t* indices, const int32_t* last_page_len,
                                float sm_scale, void* out, float* lse, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * Bind `workspace` to `plan` ("Oxide Infer" README, "One execution model":
 * the plan fixes the work decomposition once and every run only enqueues;
 * "Providers": explicit workspace). Enqueues on `stream` the copy of the
 * plan's work list (units, per-CTA ranges, split-merge entries) into the
 * workspace, followed by a 64-bit stamp of the plan in its header.
 *
 * Later oxd_paged_decode_run calls of this plan that pass this same
 * workspace pointer then read the work list from the workspace: the kernels
 * are launched with small parameter blocks and the run copies nothing. Runs
 * on any other workspace are unaffected. A plan holds one binding at a time
 * (binding another workspace replaces it); destroying the plan ends it.
 *
 *   workspace       device scratch of at least the planned size, 256-byte
 *                   aligned, on the plan's device
 *   workspace_bytes its size
 *   stream          cudaStream_t; runs on other streams must be ordered
 *                   after this copy by the caller
 *
 * Ownership: from the call on, bytes [0, 256 + list size) of the workspace
 * belong to the binding. Anything else written there (another plan's run or
 * binding on the same workspace, a memset, handing the memory to another
 * user) ends it on the device: each kernel checks the stamp before it uses
 * the list, and on a mismatch computes nothing and records
 * OXD_DEVICE_PLAN_MISMATCH (read with oxd_read_device_status). Every unit
 * read from a bound list is also bounds-checked against the plan's batch,
 * heads, page count and slot count, so a damaged list is reported the same
 * way and never leads the kernels outside the caller's buffers. After the
 * memory was reused, bind again.
 *
 * Errors (nothing enqueued): OXD_ERR_INVALID_ARGUMENT (NULL),
 * OXD_ERR_ALIGNMENT, OXD_ERR_WORKSPACE_TOO_SMALL, OXD_ERR_PLAN_MISMATCH
 * (destroyed or host-only plan, or another current device), OXD_ERR_CUDA.
 */
oxd_status oxd_plan_bind_workspace(oxd_plan plan, void* workspace, size_t workspace_bytes,
                                   void* stream);

/*
 * oxd_paged_decode_run without a caller-provided workspace. The source pages
 * have no counterpart to this entry point; it exists for callers that cannot
 * call cudaMalloc: a serving process that reserves all of its device memory
 * at start-up and allows no later allocation (so memory never fragments and
 * no allocation stalls a decode step), or a host that reaches this library
 * through a plugin interface that passes only input and output tensors.
 *
 * The scratch is a 32 MiB array inside the library, reserved on every GPU
 * that loads the library and held until the process exits. The call
 * allocates nothing (no cudaMalloc, no cudaFree, no allocating library call).
 * Arguments and results are those of oxd_paged_decode_run minus the
 * workspace. A plan whose workspace_bytes exceeds 32 MiB is rejected with
 * OXD_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture. Every call on a device shares the one array,
 * which keeps the last call's contents; nothing in it has to start at zero
 * (a run writes everything it reads, and its status word is tagged with the
 * run's epoch, so what an earlier call left is never read as this call's).
 * Calls that can overlap on the GPU (other streams, other threads) race on
 * the array and must be serialised by the caller.
 * The device status word lives in that array: read it with
 * oxd_read_static_workspace_status, not oxd_read_device_status.
 */
oxd_status oxd_paged_decode_run_static_workspace(oxd_plan plan, const void* q,
                                                 const void* k_pages, const void* v_pages,
                                                 const int32_t* indptr, const int32_t* indices,
                                                 const int32_t* last_page_len, float sm_scale,
                                                 void* out, float* lse, void* stream);

/*
 * The device status of the last oxd_paged_decode_run_static_workspace call on
 * the calling thread's current device (the pages have no counterpart; it
 * completes the allocation-free entry point above, whose status word is in
 * the library's array). Synchronises `stream`, then reads into *code the
 * first error that call's kernels recorded (a page index outside the pool,
 * device tables that differ from the plan's, a wait that ran out), or
 * OXD_DEVICE_OK. Allocates nothing. Returns OXD_OK when the code is
 * OXD_DEVICE_OK, OXD_ERR_DEVICE_STATUS otherwise, OXD_ERR_INVALID_ARGUMENT
 * for a NULL `code`, OXD_ERR_CUDA if a CUDA call failed. Another static-array
 * call enqueued after the one of interest replaces the status.
 */
oxd_status oxd_read_static_workspace_status(void* stream, int32_t* code);

/*
 * Merge attention states ("Attention state and cascade": state merge).
 * For each n < N and h < H, combine the S states (v[n, i, h, :], s[n, i, h]):
 *   M = max_i s_i, w_i = exp(s_i - M),
 *   v_out[n, h, :] = sum_i w_i v_i / sum_i w_i,  s_out[n, h] = M + ln sum_i w_i.
 * States with s_i = -inf carry no weight; if all are -inf, v_out = 0 and
 * s_out = -inf. s uses the natural logarithm, as lse from a run does.
 *
 *   v      device f32 [N][S][H][D], 16-byte aligned, D % 4 == 0
 *   s      device f32 [N][S][H], 4-byte aligned
 *   v_out  device bf16 [N][H][D], 8-byte aligned
 *   s_out  device f32 [N][H] or NULL
 * Errors: OXD_ERR_INVALID_ARGUMENT (non-positive sizes, D % 4 != 0, NULL),
 * OXD_ERR_ALIGNMENT, OXD_ERR_ALIAS (outputs overlap inputs or each other),
 * OXD_ERR_CUDA.
 */
oxd_status oxd_merge_states(const float* v, const float* s, int32_t N, int32_t S, int32_t H,
                            int32_t D, void* v_out, float* s_out, void* stream);

/*
 * Fused rotary embedding and paged KV append ("FlashInfer parity matrix",
 * "Admitted attention matrix", rows "Standard RoPE" -- D128 NeoX split-half
 * with explicit int32 positions -- and "Fused RoPE plus paged append";
 * "Paged KV ownership difference": decode may read shared pages, the append
 * writes only to pages whose reference count is one, and the pager makes a
 * target page private and remaps the request before enqueue).
 *
 * Token t (t < T) belongs to request b = token_request[t] at logical
 * position p = positions[t]. With h = 64 and f_i = rope_theta^(-2i/128):
 *   RoPE(x, p)_i      = x_i cos(p f_i) - x_{i+h} sin(p f_i)
 *   RoPE(x, p)_{i+h}  = x_{i+h} cos(p f_i) + x_i sin(p f_i),   i < h
 * For every query head q_out[t] = bf16(RoPE(q[t], p)); for every KV head the
 * K row bf16(RoPE(k[t], p)) and the V row v[t] (unchanged) are written to
 * page indices[indptr[b] + p / page_size], slot p % page_size, of the pools
 * (the block table must already cover the position; positions are below
 * 2^24). The rotation runs in float with the angle carried as a two-float
 * number of turns; out-of-order tokens, several tokens
 * of one request and tokens of different requests may share a call; two
 * tokens must not target the same (page, slot).
 *
 *   desc          shapes; num_tokens >= 1, head_dim 128, page_size in
 *                 {8, 16, 32, 64}, rope_theta finite and > 1
 *   q, q_out      device bf16 [T][Hq][128], 16-byte aligned; q_out may be q
 *                 itself (in place) but must not overlap it otherwise
 *   k, v          device bf16 [T][Hkv][128], 16-byte aligned
 *   token_request, positions  device int32 [T]
 *   indptr, indices           device int32 block tables (as for decode); indices
 *                 holds desc->num_indices entries
 *   page_refcount device int32 [num_pages]: the caller's authoritative
 *                 snapshot of each page's reference count
 *   k_pages, v_pages  device bf16 pools (desc layout), written in place
 *   workspace     device, >= 256 bytes, 256-byte aligned, any contents: the
 *                 status word, read with oxd_read_device_status
 *   stream        cudaStream_t
 * Host-side errors (nothing enqueued): OXD_ERR_INVALID_ARGUMENT,
 * OXD_ERR_UNSUPPORTED, OXD_ERR_ALIGNMENT, OXD_ERR_ALIAS (an output overlaps
 * an input or another output, other than q_out == q),
 * OXD_ERR_WORKSPACE_TOO_SMALL, OXD_ERR_CUDA. Device-side: a token whose
 * request or position lies outside the block table
 * (OXD_DEVICE_BAD_POSITION), whose page index lies outside the pool
 * (OXD_DEVICE_BAD_PAGE) or whose page is shared (OXD_DEVICE_SHARED_PAGE)
 * writes no K/V row; the other tokens are written, and every q_out row is. A
 * request whose indptr entries are negative, decreasing or past num_indices,
 * or a position outside [0, 2^24), counts as OXD_DEVICE_BAD_POSITION; such a
 * token's q_out rows are rotated at position p & (2^24 - 1).
 */
typedef struct {
    int32_t num_tokens;     /* T */
    int32_t batch;          /* B: requests in the block tables */
    int32_t num_qo_heads;
    int32_t num_kv_heads;
    int32_t head_dim;       /* 128 */
    int32_t page_size;      /* 8, 16, 32 or 64 */
    int32_t layout;         /* oxd_kv_layout */
    int32_t num_indices;    /* entries of `indices` (indptr[B]); the device refuses tables
                               that point past it */
    int64_t num_pages;      /* pages in each pool and in page_refcount */
    double rope_theta;      /* frequency base (10000 in the standard variant) */
    int32_t reserved[2];    /* must be zero */
} oxd_rope_append_desc;

oxd_status oxd_rope_append(const oxd_rope_append_desc* desc, const void* q, const void* k,
                           const void* v, const int32_t* token_request, const int32_t* positions,
                           const int32_t* indptr, const int32_t* indices,
                           const int32_t* page_refcount, void* q_out, void* k_pages,
                           void* v_pages, void* workspace, size_t workspace_bytes,
                           void* stream);

/*
 * Paged causal prefill ("FlashInfer parity matrix" page, "Admitted attention
 * matrix", row "Paged causal prefill": BF16, D128, causal, over the same
 * NHD/HND pages and block tables as decode, long ranges split into pieces
 * with a caller-owned F32 workspace; "Domain coverage", "Prefill attention").
 *
 * Request b has L_b cached tokens (its block table, as for decode) and
 * q_len_b = qo_indptr[b+1] - qo_indptr[b] query tokens, which are the last
 * q_len_b of its cached tokens (their K and V are already in the pages, e.g.
 * written by oxd_rope_append). Query token i of request b (global index
 * qo_indptr[b] + i) sits at position p = L_b - q_len_b + i and, for each
 * query head hq (KV head hq / G, G = Hq / Hkv), computes
 *   s_j = sm_scale * q . k_j (j = 0 .. p),  out = softmax(s) V,
 *   lse = ln sum_j exp(s_j).
 * Numerics as for decode: F32 softmax state, QK^T and PV on the tensor cores
 * with BF16 operands (P rounded to BF16), out rounded once to BF16.
 *
 * Lifecycle as for decode ("Oxide Infer" README, "One execution model"): a
 * host-side plan fixes the tiles (up to tile_rows / G query tokens of one
 * request with the G heads of one KV head: 256-row tiles in two halves of
 * 128, one CTA a SM, 128-token stages; or 128-row tiles, two CTAs a SM,
 * 64-token stages), the pieces of long tiles and the workspace size; runs
 * only check operands and enqueue.
 */
typedef struct oxd_prefill_plan_s* oxd_prefill_plan;

typedef struct {
    int32_t batch;          /* B requests */
    int32_t num_qo_heads;   /* Hq */
    int32_t num_kv_heads;   /* Hkv; Hq % Hkv == 0, Hq / Hkv <= 128 */
    int32_t head_dim;       /* 128 */
    int32_t page_size;      /* 8, 16, 32 or 64 */
    int32_t layout;         /* oxd_kv_layout */
    int64_t num_pages;      /* pages in each pool */
    int32_t max_splits;     /* 0: the planner splits long tiles to fill the GPU;
                               1: never split; n > 1: at most n pieces per tile */
    int32_t num_sms;        /* 0: plan for the device; > 0: host-only plan for that
                               many SMs (runs refused) */
    int64_t wait_timeout_ns; /* limit of one pipeline wait, as for decode: 0 = about one
                                second, n > 0 = n nanoseconds */
    int32_t tile_rows;      /* 0: the planner picks (128 when a plan of 256-row tiles
                               would give fewer 128-token stages than the GPU has SMs,
                               else 256); 128 or 256: that tile size; other values are
                               OXD_ERR_INVALID_ARGUMENT */
    int32_t reserved;       /* must be zero */
} oxd_paged_prefill_desc;

typedef struct {
    int32_t tile_tokens;        /* query tokens per tile: tile_rows / G */
    int32_t num_tiles;
    int32_t num_units;          /* CTAs per run: pieces of all tiles */
    int32_t num_split_tiles;
    int32_t max_pieces;
    int32_t num_merge_rows;     /* output rows merged from pieces (0: one launch) */
    int32_t launches_per_run;   /* 1, or 2 with the merge */
    int32_t ctas_per_sm;
    int32_t num_sms;
    int32_t tile_rows;          /* 128 or 256: the tile size (and kernel) the plan runs */
    int64_t workspace_bytes;
    int64_t total_q_tokens;
    int64_t total_kv_tokens;
    int64_t causal_pairs;       /* (query token, cached token) pairs per query head */
} oxd_prefill_plan_info;

/*
 * Plan a prefill over host copies of the tables.
 *   qo_indptr      host int32 [B+1], qo_indptr[0] = 0, non-decreasing
 *   indptr         host int32 [B+1] (at least one page per request)
 *   last_page_len  host int32 [B], in [1, page_size]
 *   device         CUDA device the plan is for (ignored for a host-only plan)
 * q_len_b must not exceed L_b; a request with q_len_b = 0 adds no work, but
 * the batch needs at least one query token.
 * Writes the plan and its workspace size. Errors: OXD_ERR_INVALID_ARGUMENT,
 * OXD_ERR_UNSUPPORTED (head_dim, page size, group size), OXD_ERR_CUDA,
 * OXD_ERR_NO_MEMORY.
 */
oxd_status oxd_paged_prefill_plan(const oxd_paged_prefill_desc* desc, const int32_t* qo_indptr,
                                  const int32_t* indptr, const int32_t* last_page_len,
                                  int device, oxd_prefill_plan* plan_out,
                                  size_t* workspace_bytes);

/*
 * Enqueue one prefill on `stream`.
 *   q              device bf16 [Nq][Hq][128], Nq = qo_indptr[B], 16-byte aligned
 *   k_pages, v_pages  device bf16 pools (desc layout), 16-byte aligned
 *   qo_indptr, indptr, indices, last_page_len  device int32 tables equal to
 *                  the ones planned (indices may differ: page contents are
 *                  read through them at run time)
 *   sm_scale       finite
 *   out            device bf16 [Nq][Hq][128], 16-byte aligned
 *   lse            device f32 [Nq][Hq] or NULL
 *   workspace      device scratch of the planned size, 256-byte aligned
 * Unless the workspace is bound to the plan (oxd_prefill_plan_bind_workspace),
 * the run first copies the plan's work list into it. Errors (nothing
 * enqueued): OXD_ERR_INVALID_ARGUMENT, OXD_ERR_ALIGNMENT, OXD_ERR_ALIAS,
 * OXD_ERR_WORKSPACE_TOO_SMALL, OXD_ERR_PLAN_MISMATCH (destroyed or host-only
 * plan, other device), OXD_ERR_CUDA. Device-side: an out-of-range page index
 * (read as page 0), device tables that differ from the plan's, a damaged
 * bound list or a wait timeout are recorded in the workspace status word.
 */
oxd_status oxd_paged_prefill_run(oxd_prefill_plan plan, const void* q, const void* k_pages,
                                 const void* v_pages, const int32_t* qo_indptr,
                                 const int32_t* indptr, const int32_t* indices,
                                 const int32_t* last_page_len, float sm_scale, void* out,
                                 float* lse, void* workspace, size_t workspace_bytes,
                                 void* stream);

/* As oxd_plan_bind_workspace, for a prefill plan: later runs on this
 * workspace read the work list from it and copy nothing. */
oxd_status oxd_prefill_plan_bind_workspace(oxd_prefill_plan plan, void* workspace,
                                           size_t workspace_bytes, void* stream);
/* As oxd_plan_set_timing_events: events recorded around the prefill kernel. */
oxd_status oxd_prefill_plan_set_timing_events(oxd_prefill_plan plan, void* event_before,
                                              void* event_after);
oxd_status oxd_prefill_plan_get_info(oxd_prefill_plan plan, oxd_prefill_plan_info* info);
oxd_status oxd_prefill_plan_destroy(oxd_prefill_plan plan);

/* Planner decisions of a plan (host only). */
oxd_status oxd_plan_get_info(oxd_plan plan, oxd_plan_info* info);

/*
 * Record caller-created CUDA events immediately before and after the decode
 * kernel of every later run of this plan (cudaEvent_t values; NULL, NULL
 * turns it off). For measuring the kernel alone; the plan is otherwise
 * unchanged.
 */
oxd_status oxd_plan_set_timing_events(oxd_plan plan, void* event_before, void* event_after);

/*
 * Release a plan. Only after every run that used it has completed on the GPU
 * (its page-locked work list may still be being copied until then; the
 * "Providers" section's completion-owned lease).
 */
oxd_status oxd_plan_destroy(oxd_plan plan);

/*
 * Synchronise `stream`, then read into *code the first error the last run
 * that started on `workspace` recorded (OXD_DEVICE_OK if it recorded none). Returns OXD_OK when
 * the code is OXD_DEVICE_OK, OXD_ERR_DEVICE_STATUS otherwise, OXD_ERR_CUDA if
 * the copy failed. This is the one call that blocks the host.
 */
oxd_status oxd_read_device_status(const void* workspace, void* stream, int32_t* code);

/* Static strings for a status and a device status code. */
const char* oxd_status_string(oxd_status status);
const char* oxd_device_status_string(int32_t code);

/* Library version string, e.g. "oxd 0.1.0 sm_103a". */
const char* oxd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* OXD_H */
