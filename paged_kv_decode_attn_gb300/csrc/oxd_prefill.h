// Internal declarations of the paged causal prefill (kernel and host side).
// Not part of the public ABI (include/oxd.h is).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace oxd {

constexpr int kPrefillRows = 256;         // rows of a tile: tile_tokens * G (<= 256), two
                                          // halves of 128 MMA rows
constexpr int kMaxPrefillGroup = 128;     // G = Hq / Hkv of a prefill
constexpr int kPrefillStageTokens = 128;  // cached tokens per pipeline stage
// The narrow kernel (short prefills and the cascade decode's shared-prefix
// tiles): 128-row tiles on 64-token stages, two CTAs a SM.
constexpr int kNarrowRows = 128;
constexpr int kNarrowStageTokens = 64;

// One CTA's work: a piece of the cached-token range of one tile (up to
// tile_tokens consecutive query tokens of one request, with the G query heads
// of one KV head each). 64 bytes.
struct PrefillUnit {
    int32_t idx_begin;  // offset in `indices` of the piece's first page
    int32_t n_pages;    // pages the piece reads
    int32_t kv_begin;   // first cached token of the piece (a multiple of 128)
    int32_t kv_valid;   // cached tokens of the piece, >= 1
    int32_t q_begin;    // global index of the tile's first query token
    int32_t n_tok;      // query tokens of the tile, 1 .. tile_tokens
    int32_t p0;         // position of the tile's first query token in its request
    int32_t hkv;        // KV head
    int32_t b;          // request
    int32_t state;      // split tile: state group of its token 0 (token t, piece i
                        // -> group state + t * n_pieces + i); unused when unsplit
    int32_t n_pieces;   // pieces of the tile (1: the CTA writes out/lse itself)
    int32_t piece;      // this piece's index
    int32_t qo_b;       // qo_indptr[b], L_b and indptr[b] as planned: the
    int32_t kv_len;     // kernel checks the device tables against them
    int32_t page_base;
    int32_t pad;
};
static_assert(sizeof(PrefillUnit) == 64, "units are 64 bytes");

struct PrefillParams {
    const uint16_t* q;              // bf16 [Nq][Hq][128]
    uint16_t* out;                  // bf16 [Nq][Hq][128]
    float* lse;                     // [Nq][Hq] or nullptr
    const int32_t* qo_indptr;       // nullptr: rows are not checked against one (cascade)
    const int32_t* indptr;
    const int32_t* indices;
    const int32_t* last_page_len;
    const PrefillUnit* units;       // in the workspace
    const unsigned long long* ws_stamp;  // bound workspace: its stamp word, else nullptr
    unsigned long long stamp;
    unsigned long long* clear_stamp;     // unbound run: the stamp word, set to 0
    float* part_o;                  // f32 [groups][G][128]
    float* part_lse;                // f32 [groups][G] (log2)
    int64_t n_states;               // groups * G
    unsigned long long* status;
    uint32_t* last_epoch;
    uint32_t epoch;
    int32_t n_units;
    int32_t batch;
    int32_t n_q_tokens;
    int64_t nnz;
    int32_t num_qo_heads;
    int32_t num_kv_heads;
    int32_t group;
    int32_t tile_tokens;
    int32_t page_size;
    int32_t layout;
    int64_t num_pages;
    float scale_log2;
    int32_t wait_prior;             // 1: launched early behind another grid, which must
                                    // complete before this one does (griddepcontrol.wait)
    int64_t wait_ns;                // limit of a pipeline wait (> 0)
};

cudaError_t prefill_smem_bytes(int* bytes);
cudaError_t prefill_occupancy(int* ctas_per_sm);
// tk, tv: the pool maps (as for decode).
// early: launched with programmatic dependent launch behind the previous
// kernel on the stream (then p.wait_prior must be 1).
cudaError_t launch_prefill(const CUtensorMap& tk, const CUtensorMap& tv, const PrefillParams& p,
                           int grid, cudaStream_t stream, bool early = false);
cudaError_t prefill_narrow_smem_bytes(int* bytes);
cudaError_t prefill_narrow_occupancy(int* ctas_per_sm);
// The narrow kernel: tiles of at most kNarrowRows rows, pieces starting at a
// multiple of kNarrowStageTokens; tq: q as (d, head, token) with a box of
// 64 x G x (kNarrowRows / G) and the 128-byte swizzle.
cudaError_t launch_prefill_narrow(const CUtensorMap& tk, const CUtensorMap& tv,
                                  const CUtensorMap& tq, const PrefillParams& p, int grid,
                                  cudaStream_t stream, bool early = false);

}  // namespace oxd
