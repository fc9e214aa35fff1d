// Internal declarations shared by the library's host code and its kernels.
// Not part of the public ABI (include/oxd.h is).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace oxd {

constexpr int kHeadDim = 128;
constexpr int kMaxGroup = 32;           // G = Hq / Hkv handled by the decode kernels
constexpr int kSliceTokens = 16;        // tokens one consumer warp handles per stage
constexpr long long kWaitTimeoutNs = 1000000000LL;  // bounded waits (1 s)

// Decode kernel variants (oxd_plan_info.kernel_variant).
enum Variant : int {
    kVariantFmaG1 = 0,   // CUDA-core FMA, G = 1 (MHA)
    kVariantFmaG2 = 1,   // CUDA-core FMA, G = 2
    kVariantMma8 = 2,    // mma.sync m16n8k16, 3 <= G <= 8 (rows 8..15 of the tile idle)
    kVariantMma16 = 3,   // mma.sync, 9 <= G <= 16
    kVariantMma32 = 4,   // mma.sync, two 16-row tiles, 17 <= G <= 32
    kNumVariants = 5
};

struct VariantShape {
    int threads;        // consumer warps * 32 + one producer warp
    int stage_tokens;   // tokens per pipeline stage
    int stages;         // pipeline depth
    int smem_bytes;     // dynamic shared memory per CTA
};

// One work item: consecutive pages of one request, processed once per KV
// head (a work unit is an (item, KV head) pair; unit u = item u / Hkv, head
// u % Hkv). The planned indptr/last_page_len of the request ride along so the
// kernel can check the device block tables against the plan.
struct WorkItem {
    int32_t idx_begin;   // absolute offset of the item's first page in `indices`
    int32_t n_pages;
    int32_t valid;       // valid tokens in the item (the last page may be partial)
    int32_t b;           // request
    int32_t slot;        // partial-state slot, or -1: the item is its whole request
    int32_t indptr_b;    // planned indptr[b], indptr[b+1], last_page_len[b]
    int32_t indptr_b1;
    int32_t last;
};
static_assert(sizeof(WorkItem) == 32, "work item is 32 bytes");

// Work lists up to this length travel in the decode kernel's parameter
// buffer; longer ones are copied into the workspace.
constexpr int kInlineItems = 448;
struct InlineWork {
    WorkItem item[kInlineItems];
};

// Split requests, {b, first slot, slots, 0}; same rule for the merge kernel.
constexpr int kInlineSplits = 1024;
struct InlineSplits {
    int4 split[kInlineSplits];
};

// Workspace layout (byte offsets, each 256-aligned):
//   [0, 256)     header: int32 status word, int32 work counter (the run
//                zeroes both with a 16-byte memset before the decode kernel)
//   items        WorkItem[n_items]   (written by the run only when too long
//   split        int4[n_split]        for the parameter buffers)
//   part_o       f32[n_slots][Hq][128]
//   part_lse     f32[n_slots][Hq]  (log2 domain)
struct WsHeader {
    int32_t status;
    int32_t work_counter;
    int32_t pad[62];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

struct DecodeParams {
    const uint16_t* q;            // bf16 [B][Hq][128]
    uint16_t* out;                // bf16 [B][Hq][128]
    float* lse;                   // [B][Hq] or nullptr
    const int32_t* indptr;
    const int32_t* indices;
    const int32_t* last_page_len;
    const WorkItem* items;        // nullptr: the work list is the InlineWork parameter
    float* part_o;
    float* part_lse;
    int32_t* status;
    int32_t* work_counter;
    int32_t num_qo_heads;
    int32_t num_kv_heads;
    int32_t group;                // G
    int32_t page_size;
    int32_t layout;               // 0 NHD, 1 HND
    int32_t n_units;              // n_items * num_kv_heads
    int64_t num_pages;
    float scale_log2;             // sm_scale * log2(e)
};

struct MergeParams {
    const float* v;               // states [.][H][D], state-major
    const float* s;               // [.][H]
    uint16_t* out;                // bf16 [rows][H][D]
    float* lse;                   // [rows][H] natural log, or nullptr
    const int4* split;            // split table in memory; nullptr: inline (split mode)
    int32_t split_mode;           // 1: row n is split[n] = {row, first state, count, 0};
                                  // 0: row n uses states [n*S, n*S + S)
    int32_t n;                    // rows to merge
    int32_t S;                    // states per row when split_mode == 0
    int32_t H;
    int32_t D;
    float s_to_ln;                // factor taking s to natural log (1, or ln 2 for log2)
};

// Implemented in oxd_decode.cu / oxd_merge.cu.
VariantShape variant_shape(int variant);
cudaError_t variant_occupancy(int variant, int* ctas_per_sm);
cudaError_t launch_decode(int variant, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                          const DecodeParams& p, const InlineWork& work, int grid,
                          cudaStream_t stream);
// Uniform-state merge (the public entry point).
cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream);
// Merge of the split requests of a decode run, launched behind the decode
// kernel with programmatic dependent launch when `early` (it waits for the
// decode grid before reading anything).
cudaError_t launch_split_merge(const MergeParams& p, const InlineSplits& splits,
                               cudaStream_t stream, bool early);

}  // namespace oxd
