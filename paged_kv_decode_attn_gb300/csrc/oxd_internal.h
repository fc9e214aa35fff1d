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
constexpr long long kWaitTimeoutNs = 1000000000LL;  // bounded pipeline waits (1 s)

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

// Work list entry, one per (request, chunk of consecutive pages).
//   x: absolute offset of the chunk's first page in `indices`
//   y: pages in the chunk
//   z: valid tokens in the chunk (the last page of a request may be partial)
//   w: request index b
// A parallel int32 array gives the partial-state slot of each item, or -1
// when the item covers its whole request and writes out/lse directly.
//
// Per-request table (int4): x = indptr[b], y = indptr[b+1], z = last_page_len[b]
// as planned (the kernels compare them with the device block tables), w = 0.
// Split-request table (int4): x = b, y = first slot, z = number of slots, w = 0.
//
// Workspace layout (byte offsets, each 256-aligned), all written by the
// run's single host-to-device copy except the partial states:
//   [0, 256)         header: int32 status word, then plan facts
//   items            int4[n_items]
//   item_slot        int32[n_items]
//   req              int4[B]
//   split            int4[n_split]
//   part_o           f32[n_slots][Hq][128]   (not uploaded)
//   part_lse         f32[n_slots][Hq]        (not uploaded)
struct WsHeader {
    int32_t status;
    int32_t n_items;
    int32_t batch;
    int32_t num_kv_heads;
    int32_t pad[60];
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
    const int32_t* item_slot;
    const int4* req;
    float* part_o;
    float* part_lse;
    int32_t* status;
    int32_t num_qo_heads;
    int32_t num_kv_heads;
    int32_t group;                // G
    int32_t page_size;
    int32_t layout;               // 0 NHD, 1 HND
    int32_t n_items;
    int64_t num_pages;
    float scale_log2;             // sm_scale * log2(e)
};

struct MergeParams {
    const float* v;               // states [.][S][H][D] (slot-major)
    const float* s;               // [.][S][H]
    uint16_t* out;                // bf16 [N][H][D]
    float* lse;                   // [N][H] or nullptr
    const int4* split;            // ragged mode: {b, first state, count, 0}; nullptr: uniform
    int32_t n;                    // number of (request) rows
    int32_t S;                    // uniform state count
    int32_t H;
    int32_t D;
};

// Implemented in oxd_decode.cu / oxd_merge.cu.
VariantShape variant_shape(int variant);
cudaError_t variant_occupancy(int variant, int* ctas_per_sm);
cudaError_t launch_decode(int variant, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                          const DecodeParams& p, int grid, cudaStream_t stream);
cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream);

}  // namespace oxd
