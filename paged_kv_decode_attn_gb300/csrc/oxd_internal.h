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
constexpr int kMaxClusterCtas = 8;                  // CTAs of a merging cluster (portable size)

// Decode kernel variants (oxd_plan_info.kernel_variant).
enum Variant : int {
    kVariantFmaG1 = 0,   // CUDA-core FMA, G = 1 (MHA)
    kVariantFmaG2 = 1,   // CUDA-core FMA, G = 2
    kVariantMma8 = 2,    // mma.sync m16n8k16, 3 <= G <= 8 (rows 8..15 of the tile idle)
    kVariantMma16 = 3,   // mma.sync, 9 <= G <= 16
    kVariantMma32 = 4,   // 17 <= G <= 32: each piece runs on a pair of 16-row CTAs
    kVariantWide = 5,    // 17 <= G <= 32: tcgen05 (TMEM accumulators), one CTA per piece
    kNumVariants = 6
};

struct VariantShape {
    int threads;        // consumer warps * 32 + one producer warp
    int stage_tokens;   // tokens per pipeline stage
    int stages;         // pipeline depth
    int smem_bytes;     // dynamic shared memory per CTA
};

// One work unit: consecutive pages of one request for one KV head.
//   x: absolute offset of the unit's first page in `indices`
//   y: pages (bits 0..23); bits 24..30: the request's last_page_len when the
//      unit ends at the request's last page, else 0; bit 31: the unit starts
//      at the request's first page
//   z: request b (bits 0..18) | second 16-row half of a G > 16 group (bit 19)
//      | KV head (bits 20..31)
//   w: partial-state slot, or -1 when the unit is its whole (request, head)
// The planner cuts the concatenation of all (request, KV head) page streams
// into one contiguous share per CTA; CTA c runs units
// [cta_begin[c], cta_begin[c+1]) in order.
constexpr int kUnitPagesBits = 24;
constexpr int kUnitBBits = 19;

struct WorkList {
    static constexpr int kUnits = 1728;  // units carried in the parameter buffer
    static constexpr int kCtas = 600;    // CTA ranges carried in the parameter buffer
    int4 unit[kUnits];
    int32_t cta_begin[kCtas + 1];
};

// Per split (request, KV head): x = first output row (b*Hq + hkv*G),
// y = first slot, z = slots, w = 0.
struct SplitList {
    static constexpr int kEntries = 1024;
    int4 entry[kEntries];
};

// Workspace layout (byte offsets, each 256-aligned):
//   [0, 256)     header: status word {epoch, code} of the last run that
//                recorded an error, the epoch of the last run that started,
//                and the stamp of the plan bound to the workspace
//   (a bound workspace holds the units, CTA ranges and merge entries for
//   good; runs on it pass no work list and copy nothing)
//   units        int4[n_units]        \ written by oxd_plan_bind_workspace, or
//   cta_rec      int4[grid][2]         > by an unbound run whose list does not
//   splits       int4[n_split]        /  fit the kernels' parameter buffers
// cta_rec[c] = {first unit, end unit, 0, 0}, then a copy of the CTA's first
// unit, so one 32-byte load starts the CTA.
//   part_o       f32[n_slots][G][128]
//   part_lse     f32[n_slots][G]  (log2 domain)
struct WsHeader {
    unsigned long long status;
    uint32_t last_epoch;
    uint32_t pad0;
    unsigned long long stamp;      // plan stamp of a bound workspace (oxd_plan_bind_workspace)
    uint32_t pad[58];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

struct DecodeParams {
    const uint16_t* q;            // bf16 [B][Hq][128]
    uint16_t* out;                // bf16 [B][Hq][128]
    float* lse;                   // [B][Hq] or nullptr
    const int32_t* indptr;
    const int32_t* indices;
    const int32_t* last_page_len;
    const int4* units;            // nullptr: the WorkList parameter holds the units
    const int4* cta_rec;          //          and the CTA ranges
    const unsigned long long* ws_stamp;  // bound workspace: its stamp word, else nullptr
    unsigned long long stamp;            // the plan's stamp
    unsigned long long* clear_stamp;     // unbound run: the workspace's stamp word, set to 0
    int32_t n_units;              // bounds every unit is checked against
    int32_t n_slots;
    int32_t batch;
    int32_t pad0;
    int64_t nnz;
    float* part_o;
    float* part_lse;
    unsigned long long* status;
    uint32_t* last_epoch;
    uint32_t epoch;               // this run's epoch (never 0)
    int32_t num_qo_heads;
    int32_t num_kv_heads;
    int32_t group;                // G
    int32_t page_size;
    int32_t layout;               // 0 NHD, 1 HND
    int64_t num_pages;
    float scale_log2;             // sm_scale * log2(e)
    // > 1: launched as clusters of this many CTAs, one stream per cluster,
    // piece r on rank r (slot = CTA index); rank 0 merges the cluster's
    // partial states into out/lse. 0: no cluster merge.
    int32_t cluster_c;
    int32_t pad1;
    int64_t wait_ns;              // limit of a pipeline wait (> 0)
};

// Merge of R-row states. Entry n: output rows first_row + r, r < R, from
// states (first + i) * R + r, i < count (state-major [.][R][D] layout).
struct MergeParams {
    const float* v;               // states [.][R][D]
    const float* s;               // [.][R]
    uint16_t* out;                // bf16 rows of D
    float* lse;                   // per output row, natural log, or nullptr
    const unsigned long long* ws_stamp;  // bound workspace: its stamp word, else nullptr
    unsigned long long stamp;
    int64_t n_rows;               // output rows (entries are checked against it)
    int64_t n_states;             // states available (likewise)
    const int4* entries;          // {first_row, first, count, 0}; nullptr: the
                                  // SplitList parameter (split mode) or, in
                                  // uniform mode, entry n = {n*R, n*S, S}
    int32_t uniform;              // 1: entries implicit from S
    int32_t n;                    // entries
    int32_t S;                    // states per entry in uniform mode
    int32_t R;                    // rows per entry
    int32_t D;
    float s_to_ln;                // factor taking s to natural log (1, or ln 2 for log2)
    int32_t max_count;            // most states of any entry: rows of more than 16 states
                                  // (D = 128) are merged by two warps, half a row each
};

// Fused RoPE + paged append (oxd_append.cu).
struct AppendParams {
    const uint16_t* q;            // bf16 [T][Hq][128]
    const uint16_t* k;            // bf16 [T][Hkv][128]
    const uint16_t* v;
    const int32_t* token_request; // [T]
    const int32_t* positions;     // [T]
    const int32_t* indptr;        // [B+1]
    const int32_t* indices;
    const int32_t* refcount;      // [num_pages]
    uint16_t* q_out;              // bf16 [T][Hq][128]
    uint16_t* k_pages;
    uint16_t* v_pages;
    unsigned long long* status;
    uint32_t* last_epoch;
    uint32_t epoch;
    int32_t T, B, Hq, Hkv, page_size, layout, num_indices;
    int64_t num_pages;
    float turns_hi[kHeadDim / 2];  // theta^(-2i/128) / (2 pi) as hi + lo floats
    float turns_lo[kHeadDim / 2];
};
cudaError_t launch_rope_append(const AppendParams& p, cudaStream_t stream);
// Run epochs (oxd_host.cpp): never 0, increasing over the process.
uint32_t next_run_epoch();

// Implemented in oxd_decode.cu / oxd_merge.cu.
VariantShape variant_shape(int variant);
cudaError_t variant_occupancy(int variant, int* ctas_per_sm);
// `work` == nullptr: the units live in memory (p.units), and the kernel is
// launched with a small parameter block. pdl: launched as a programmatic
// dependent of the kernel before it on the stream.
cudaError_t launch_decode(int variant, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                          const DecodeParams& p, const WorkList* work, int grid,
                          cudaStream_t stream, bool pdl);
// The tcgen05 variant for groups of 17..32 query heads (oxd_decode_wide.cu);
// `tq` maps q as [B*Hq rows][128] with the 128-byte swizzle.
VariantShape wide_shape();
cudaError_t wide_occupancy(int* ctas_per_sm);
cudaError_t launch_decode_wide(const CUtensorMap& tk, const CUtensorMap& tv,
                               const CUtensorMap& tq, const DecodeParams& p, const WorkList* w,
                               int grid, cudaStream_t stream, bool pdl);
// Uniform-state merge (the public entry point).
cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream);
// Merge of the split (request, KV head) streams of a decode run, launched
// behind the decode kernel with programmatic dependent launch when `early`
// (it waits for the decode grid before reading anything).
cudaError_t launch_split_merge(const MergeParams& p, const SplitList* splits,
                               cudaStream_t stream, bool early);

// Empty stand-in for the parameter-buffer lists of a bound run.
struct NoList {
    int32_t unused;
};

}  // namespace oxd
