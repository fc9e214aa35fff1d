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
    int64_t num_pages;
    float scale_log2;             // sm_scale * log2(e)
};

struct MergeParams {
    const float* v;               // states [N][S][H][D]
    const float* s;               // [N][S][H], natural log
    uint16_t* out;                // bf16 [N][H][D]
    float* lse;                   // [N][H] or nullptr
    int32_t n;
    int32_t S;
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
