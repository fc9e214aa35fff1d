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

// Work list, two int4 per item (one item = consecutive pages of one request,
// processed once per KV head):
//   A: x = absolute offset of the item's first page in `indices`,
//      y = pages in the item, z = valid tokens in the item, w = request b
//   B: x = partial-state slot of this item or -1 when the item covers its
//      whole request (then it writes out/lse directly), y = first slot of the
//      request's items, z = number of items of the request, w = 0
// Per-request table (int4): x = indptr[b], y = indptr[b+1], z = last_page_len[b]
// as planned (the kernel compares them with the device block tables), w = 0.
//
// Workspace layout (byte offsets, each 256-aligned); everything before
// part_o is written by the run's single host-to-device copy, which also
// zeroes the status word and all counters:
//   [0, 256)     header: int32 status word, int32 work counter
//   items        int4[2 * n_items]
//   req          int4[B]
//   counters     int32[B * Hkv]   finished items per (request, KV head)
//   split        int4[n_split]    {b, first slot, slots, 0} per split request
//                                 (read by the separate merge kernel)
//   part_o       f32[n_slots][Hq][128]
//   part_lse     f32[n_slots][Hq]  (log2 domain)
struct WsHeader {
    int32_t status;
    int32_t work_counter;
    int32_t n_items;
    int32_t batch;
    int32_t num_kv_heads;
    int32_t pad[59];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

struct DecodeParams {
    const uint16_t* q;            // bf16 [B][Hq][128]
    uint16_t* out;                // bf16 [B][Hq][128]
    float* lse;                   // [B][Hq] or nullptr
    const int32_t* indptr;
    const int32_t* indices;
    const int32_t* last_page_len;
    const int4* items;
    const int4* req;
    int32_t* counters;
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
    int32_t fused_merge;          // 1: last unit of a split request merges; 0: merge kernel
    int64_t num_pages;
    float scale_log2;             // sm_scale * log2(e)
};

struct MergeParams {
    const float* v;               // states [.][H][D], state-major
    const float* s;               // [.][H]
    uint16_t* out;                // bf16 [rows][H][D]
    float* lse;                   // [rows][H] natural log, or nullptr
    const int4* split;            // per merged row {row, first state, count, 0}; nullptr:
                                  // row n uses states [n*S, n*S + S)
    int32_t n;                    // rows to merge
    int32_t S;                    // states per row when split == nullptr
    int32_t H;
    int32_t D;
    float s_to_ln;                // factor taking s to natural log (1, or ln 2 for log2)
};

// Implemented in oxd_decode.cu / oxd_merge.cu.
VariantShape variant_shape(int variant);
cudaError_t variant_occupancy(int variant, int* ctas_per_sm);
cudaError_t launch_decode(int variant, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                          const DecodeParams& p, int grid, cudaStream_t stream);
// `after_decode`: launched behind the decode kernel with programmatic
// dependent launch (the kernel waits for the decode grid before reading).
cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream, bool after_decode);

}  // namespace oxd
