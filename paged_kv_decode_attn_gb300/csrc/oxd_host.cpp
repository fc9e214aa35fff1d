// Host side of the C ABI: planning, operand checks and enqueue.
//
// Lifecycle from the "Oxide Infer" README, "One execution model": the plan
// fixes the kernel variant, the chunking of every request's pages, the launch
// shape and the workspace contract; a run only checks operands and enqueues
// the decode kernel, whose work list rides in its parameter buffer (long
// lists are copied into the workspace first) or, once the plan has been
// bound to the workspace, is read from it, and, when some stream was split,
// a merge kernel launched right behind it. "Providers": checked span, alignment, alias and capacity rules;
// explicit workspace; caller stream; typed device status.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <functional>
#include <cmath>
#include <cstdlib>
#include <cstddef>
#include <cstring>
#include <mutex>
#include <new>
#include <random>
#include <unordered_set>
#include <vector>

#include "../../include/oxd.h"
#include "oxd_host_util.h"
#include "oxd_internal.h"
#include "oxd_prefill.h"

using namespace oxd;

struct oxd_plan_s {
    oxd_paged_decode_desc desc;
    int device;  // -1 for a host-only plan (desc.num_sms given)
    int group;
    int variant;
    int n_items;
    int n_slots;
    int n_split;
    int max_chunks;
    int chunk_pages;
    int ctas_per_sm;
    int num_sms;
    int64_t nnz;
    int64_t total_tokens;
    int grid;
    bool upload;  // work list or split table too long for the parameter buffers
    size_t off_units, off_cta, off_split, off_punits, off_part_o, off_part_lse;
    // cascade: prefix tiles run by the prefill kernel before the decode kernel
    int casc_units;
    int cluster_c;  // > 0: streams cut into this many pieces, merged inside the decode launch
    int casc_requests;
    int casc_tile_tokens;
    int64_t shared_kv;
    size_t meta_bytes, ws_bytes;
    WorkList* work;
    SplitList* splits;
    void* meta;   // host image of workspace bytes [0, meta_bytes), then the stamp
    bool pinned;
    unsigned long long stamp;             // identifies the plan in a bound workspace
    std::atomic<const void*> bound_ws;    // workspace bound by oxd_plan_bind_workspace
    cudaEvent_t ev_before;
    cudaEvent_t ev_after;
};

namespace {


// Run epochs: never 0 and increasing over the process, so a status word left
// in a workspace by an earlier run never passes for a later run's.
std::atomic<uint32_t> g_epoch{0};
uint32_t next_epoch() {
    uint32_t e = g_epoch.fetch_add(1, std::memory_order_relaxed) + 1;
    while (e == 0) e = g_epoch.fetch_add(1, std::memory_order_relaxed) + 1;
    return e;
}

// Cost of one more work unit on a CTA (its epilogue and the refill of the
// pipeline behind it), in tokens of streaming at a CTA's share of HBM
// bandwidth, per kernel variant; measured from per-CTA timelines (about
// 1.2 us for the 8-row tensor-core variant, 3 to 5 us for the paired 16-row
// CTAs, whose epilogue writes 16 rows of partial state).
double unit_overhead_tokens(int variant) {
    switch (variant) {
        case kVariantMma16: return 96.0;
        case kVariantMma32: return 320.0;
        case kVariantWide: return 96.0;
        default: return 64.0;
    }
}

// Plan stamps: a per-process random high half and a counter, never 0, so a
// stamp left in reused memory by another process or an earlier plan is not
// taken for a live plan's.
unsigned long long next_stamp() {
    static const unsigned long long hi = [] {
        std::random_device rd;
        return (static_cast<unsigned long long>(rd()) << 32);
    }();
    static std::atomic<uint32_t> counter{0};
    uint32_t c = counter.fetch_add(1, std::memory_order_relaxed) + 1;
    while (c == 0) c = counter.fetch_add(1, std::memory_order_relaxed) + 1;
    return hi | c;
}

std::mutex g_plans_mu;
std::unordered_set<oxd_plan> g_plans;

bool plan_alive(oxd_plan p) {
    std::lock_guard<std::mutex> lk(g_plans_mu);
    return g_plans.count(p) != 0;
}

int choose_variant(int G, int tensor_path) {
    if (G == 1) return kVariantFmaG1;
    if (G == 2) return kVariantFmaG2;
    if (G <= 8) return kVariantMma8;
    if (G <= 16) return kVariantMma16;
    return tensor_path == 1 ? kVariantMma32 : kVariantWide;
}

// Resident CTAs per SM without a device: limited by shared memory (228 KB
// per SM on sm_100-class parts, 1 KB reserved per CTA) and threads.
int estimate_ctas_per_sm(const VariantShape& v) {
    const int by_smem = (228 * 1024) / (v.smem_bytes + 1024);
    const int by_threads = 2048 / v.threads;
    return std::max(1, std::min(by_smem, by_threads));
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encoder() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool encode_pool(CUtensorMap* map, const void* pool, const oxd_paged_decode_desc& d) {
    return encode_kv_pool(map, pool, d.layout, d.page_size, d.num_kv_heads, d.num_pages);
}

// 2-D map over q as [B*Hq rows][128] for the tcgen05 variant: a box is 32
// rows x 64 columns with the 128-byte swizzle its score MMA reads; rows past
// the end read as zeros.
bool encode_q(CUtensorMap* map, const void* q, const oxd_paged_decode_desc& d) {
    EncodeTiledFn enc = get_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d.head_dim),
                                static_cast<cuuint64_t>(d.batch) * d.num_qo_heads};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d.head_dim) * 2};
    const cuuint32_t box[2] = {64, 32};
    const cuuint32_t elem[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q), dims,
                     strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

oxd_status check_desc(const oxd_paged_decode_desc* d) {
    if (d->batch < 1 || d->num_qo_heads < 1 || d->num_kv_heads < 1 || d->head_dim < 1 ||
        d->page_size < 1 || d->num_pages < 1)
        return OXD_ERR_INVALID_ARGUMENT;
    if (d->num_qo_heads % d->num_kv_heads != 0) return OXD_ERR_INVALID_ARGUMENT;
    if (d->layout != OXD_LAYOUT_NHD && d->layout != OXD_LAYOUT_HND)
        return OXD_ERR_INVALID_ARGUMENT;
    if (d->max_splits < 0 || d->force_splits < 0 || d->num_sms < 0)
        return OXD_ERR_INVALID_ARGUMENT;
    if (d->tensor_path != 0 && d->tensor_path != 1) return OXD_ERR_INVALID_ARGUMENT;
    if ((d->pdl != 0 && d->pdl != 1) || d->wait_timeout_ns < 0) return OXD_ERR_INVALID_ARGUMENT;
    if (d->shared_prefix_tokens < 0 || d->share_group < 0) return OXD_ERR_INVALID_ARGUMENT;
    if (d->shared_prefix_tokens == 0 ? d->share_group != 0
                                     : (d->share_group < 2 || d->page_size < 1 ||
                                        d->shared_prefix_tokens % d->page_size != 0))
        return OXD_ERR_INVALID_ARGUMENT;
    if (d->head_dim != kHeadDim) return OXD_ERR_UNSUPPORTED;
    if (d->page_size != 8 && d->page_size != 16 && d->page_size != 32 && d->page_size != 64)
        return OXD_ERR_UNSUPPORTED;
    if (d->num_qo_heads / d->num_kv_heads > kMaxGroup) return OXD_ERR_UNSUPPORTED;
    if (d->num_pages >= (int64_t{1} << 31)) return OXD_ERR_UNSUPPORTED;
    if (d->batch >= (1 << kUnitBBits) || d->num_kv_heads >= (1 << (31 - kUnitBBits)))
        return OXD_ERR_UNSUPPORTED;
    return OXD_OK;
}


}  // namespace

namespace oxd {
uint32_t next_run_epoch() { return next_epoch(); }

unsigned long long next_plan_stamp() { return next_stamp(); }

bool encode_kv_pool(CUtensorMap* map, const void* pool, int layout, int page_size,
                    int num_kv_heads, int64_t num_pages) {
    EncodeTiledFn enc = get_encoder();
    if (enc == nullptr) return false;
    const cuuint64_t D = static_cast<cuuint64_t>(kHeadDim);
    const cuuint64_t ps = static_cast<cuuint64_t>(page_size);
    const cuuint64_t H = static_cast<cuuint64_t>(num_kv_heads);
    cuuint64_t dims[4], strides[3];
    cuuint32_t box[4];
    const cuuint32_t elem[4] = {1, 1, 1, 1};
    dims[0] = D;
    dims[3] = static_cast<cuuint64_t>(num_pages);
    if (layout == OXD_LAYOUT_NHD) {
        dims[1] = H;
        dims[2] = ps;
        strides[0] = D * 2;
        strides[1] = H * D * 2;
        box[1] = 1;
        box[2] = static_cast<cuuint32_t>(ps);
    } else {
        dims[1] = ps;
        dims[2] = H;
        strides[0] = D * 2;
        strides[1] = ps * D * 2;
        box[1] = static_cast<cuuint32_t>(ps);
        box[2] = 1;
    }
    strides[2] = ps * H * D * 2;
    box[0] = 64;
    box[3] = 1;
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(pool), dims,
                     strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_bf16_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides, const uint32_t* box) {
    EncodeTiledFn enc = get_encoder();
    if (enc == nullptr || rank < 1 || rank > 5) return false;
    cuuint64_t d[5], st[4];
    cuuint32_t bx[5], elem[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
        elem[i] = 1;
    }
    for (int i = 0; i + 1 < rank; ++i) st[i] = strides[i];
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank),
                     const_cast<void*>(base), d, st, bx, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}
}  // namespace oxd

extern "C" {

const char* oxd_version(void) { return "oxd 0.1.0 sm_103a"; }

const char* oxd_status_string(oxd_status s) {
    switch (s) {
        case OXD_OK: return "ok";
        case OXD_ERR_INVALID_ARGUMENT: return "invalid argument";
        case OXD_ERR_UNSUPPORTED: return "unsupported shape or option";
        case OXD_ERR_ALIGNMENT: return "pointer misaligned";
        case OXD_ERR_ALIAS: return "output overlaps an input or another output";
        case OXD_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
        case OXD_ERR_PLAN_MISMATCH: return "plan does not match this call";
        case OXD_ERR_CUDA: return "CUDA runtime call failed";
        case OXD_ERR_DEVICE_STATUS: return "kernel reported an error";
        case OXD_ERR_NO_MEMORY: return "host allocation failed";
    }
    return "unknown status";
}

const char* oxd_device_status_string(int32_t code) {
    switch (code) {
        case OXD_DEVICE_OK: return "ok";
        case OXD_DEVICE_BAD_PAGE: return "page index outside the pool";
        case OXD_DEVICE_PLAN_MISMATCH: return "device block tables differ from the plan";
        case OXD_DEVICE_WAIT_TIMEOUT: return "pipeline wait timed out";
        case OXD_DEVICE_SHARED_PAGE: return "append target page is shared (reference count not 1)";
        case OXD_DEVICE_BAD_POSITION: return "append position outside the request's block table";
    }
    return "unknown device status";
}

oxd_status oxd_paged_decode_plan(const oxd_paged_decode_desc* desc, const int32_t* indptr,
                                 const int32_t* last, int device, oxd_plan* plan_out,
                                 size_t* ws_out) {
    if (desc == nullptr || indptr == nullptr || last == nullptr || plan_out == nullptr ||
        ws_out == nullptr)
        return OXD_ERR_INVALID_ARGUMENT;
    oxd_status st = check_desc(desc);
    if (st != OXD_OK) return st;
    const oxd_paged_decode_desc& d = *desc;
    const int B = d.batch, ps = d.page_size;
    if (indptr[0] < 0) return OXD_ERR_INVALID_ARGUMENT;
    int64_t total_pages = 0, total_tokens = 0;
    for (int b = 0; b < B; ++b) {
        const int64_t P = static_cast<int64_t>(indptr[b + 1]) - indptr[b];
        if (P < 1) return OXD_ERR_INVALID_ARGUMENT;
        if (last[b] < 1 || last[b] > ps) return OXD_ERR_INVALID_ARGUMENT;
        total_pages += P;
        total_tokens += (P - 1) * ps + last[b];
    }

    const int G = d.num_qo_heads / d.num_kv_heads;
    const int variant = choose_variant(G, d.tensor_path);
    const VariantShape vs = variant_shape(variant);
    int num_sms = d.num_sms, ctas_per_sm = 0, plan_device = -1;
    if (num_sms == 0) {
        int prev = 0;
        if (cudaGetDevice(&prev) != cudaSuccess) return OXD_ERR_CUDA;
        if (cudaSetDevice(device) != cudaSuccess) return OXD_ERR_CUDA;
        cudaError_t e1 = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, device);
        cudaError_t e2 = variant_occupancy(variant, &ctas_per_sm);
        cudaSetDevice(prev);
        if (e1 != cudaSuccess || e2 != cudaSuccess || num_sms < 1) return OXD_ERR_CUDA;
        plan_device = device;
    }
    if (ctas_per_sm < 1) ctas_per_sm = estimate_ctas_per_sm(vs);

    // ---- cascade: requests of a sharing group with more than the shared
    // prefix attend the prefix together (one prefill-kernel tile per chunk of
    // up to 128 / G consecutive such requests and KV head) and decode only
    // their pages after it.
    const int H = d.num_kv_heads;
    const int prefix_pages = d.shared_prefix_tokens / ps;  // 0 without cascade
    std::vector<int> start_page(B, 0);
    struct Chunk {
        int b0, n;  // requests [b0, b0 + n)
    };
    std::vector<Chunk> chunks;
    int casc_requests = 0;
    if (prefix_pages > 0) {
        const int T = kNarrowRows / G;
        for (int g0 = 0; g0 < B; g0 += d.share_group) {
            const int g1 = std::min(B, g0 + d.share_group);
            std::vector<int> members;
            for (int b = g0; b < g1; ++b) {
                const int64_t L = static_cast<int64_t>(indptr[b + 1] - indptr[b] - 1) * ps + last[b];
                if (L > d.shared_prefix_tokens) members.push_back(b);
            }
            if (members.size() < 2) continue;
            // consecutive runs of members, cut into chunks of at most T
            // requests (rows of requests in between are computed and unused)
            for (size_t i = 0; i < members.size();) {
                const int b0 = members[i];
                size_t j = i;
                while (j + 1 < members.size() && members[j + 1] - b0 < T) ++j;
                chunks.push_back({b0, members[j] - b0 + 1});
                i = j + 1;
            }
            for (int b : members) start_page[b] = prefix_pages;
            casc_requests += static_cast<int>(members.size());
        }
    }
    auto stream_tokens = [&](int b) {  // tokens the decode kernel streams for request b
        const int64_t L = static_cast<int64_t>(indptr[b + 1] - indptr[b] - 1) * ps + last[b];
        return L - static_cast<int64_t>(start_page[b]) * ps;
    };

    // ---- partition the work
    // Work is the page streams of all (request, KV head) pairs, request-major
    // (CTAs that run at the same time then read neighbouring heads of the
    // same pages). A piece is a run of consecutive pages of one stream; a
    // stream cut into several pieces is "split" and gets one partial-state
    // slot per piece.
    const int pps = std::max(1, vs.stage_tokens / ps);  // pages per pipeline stage
    // Groups of more than 16 query heads run every piece on a pair of CTAs,
    // one per 16-row half, side by side (the second read of each page is
    // then served by L2); the partition below is over CTA pairs.
    const int copies = variant == kVariantMma32 ? 2 : 1;
    const int64_t resident = static_cast<int64_t>(num_sms) * ctas_per_sm / copies;
    auto tokens_to = [&](int b, int k) {  // tokens in pages [0, k) of request b
        const int P = indptr[b + 1] - indptr[b];
        return k >= P ? static_cast<int64_t>(P - 1) * ps + last[b] : static_cast<int64_t>(k) * ps;
    };
    struct Piece {
        int b, h, p0, p1;
    };
    std::vector<Piece> pieces;
    std::vector<int> cta_of;  // CTA index of each piece, non-decreasing after ordering
    int grid = 0;
    // How to cut a batch whose split the planner chooses. Measured on one GPU
    // (step times of small batches): a stream's pieces cost about a stage of
    // streaming (~1 us) each when a CTA runs alone, the separate merge about
    // 2.5 us, merging inside a cluster about 0.3 us.
    //  * Whole streams: when every stream can have a CTA and the longest is at
    //    most two stages and within a line-partition share plus what the merge
    //    would cost (about 160 tokens of a CTA's streaming), each stream runs
    //    whole on its own CTA: nothing to merge.
    //  * Cluster merge (groups of up to 8 heads, whose pieces' states fit rank
    //    0's shared memory): when every stream can be cut into C >= 2 pieces
    //    (C <= 8, at least a page each, as many as the resident CTAs allow),
    //    there are at most 64 streams (many small clusters launched slower),
    //    and a piece is at most four stages (the cluster instance has a
    //    shorter ring) and within a line share plus 80 tokens, stream k runs on
    //    the C CTAs of cluster k, piece r on rank r; the pieces write their
    //    final states into rank 0, which merges them: no merge launch.
    //  * Otherwise the balanced line partition below, with a merge kernel for
    //    the streams it cuts.
    int cluster_c = 0;
    bool whole_streams = false;
    if (d.force_splits == 0 && d.max_splits == 0) {
        int64_t streamed = 0, live = 0, longest = 0, min_pages = INT64_MAX;
        for (int b = 0; b < B; ++b) {
            const int64_t t = stream_tokens(b);
            streamed += t;
            if (t > 0) live += H;
            longest = std::max<int64_t>(longest, t);
            min_pages = std::min<int64_t>(min_pages, indptr[b + 1] - indptr[b] - start_page[b]);
        }
        const int64_t stage_tokens = static_cast<int64_t>(pps) * ps;
        const int64_t line_grid = std::max<int64_t>(
            1, std::min<int64_t>(resident, std::max<int64_t>(streamed * H / stage_tokens, live)));
        const double share = static_cast<double>(streamed) * H / line_grid;
        whole_streams = live <= resident && longest <= 2 * stage_tokens &&
                        static_cast<double>(longest) <= share + 160.0;
        const int64_t n_streams = static_cast<int64_t>(B) * H;
        if (!whole_streams && prefix_pages == 0 && n_streams <= 64 &&
            (variant == kVariantFmaG1 || variant == kVariantFmaG2 || variant == kVariantMma8)) {
            const int C = static_cast<int>(
                std::min<int64_t>({kMaxClusterCtas, min_pages, resident / n_streams}));
            if (C >= 2) {
                const int64_t piece = (longest + C - 1) / C;
                if (piece <= 4 * stage_tokens && static_cast<double>(piece) <= share + 80.0)
                    cluster_c = C;
            }
        }
    }
    if (cluster_c > 0) {
        // stream k = b * H + h on CTAs [k C, k C + C), piece r on rank r
        for (int b = 0; b < B; ++b) {
            const int P = indptr[b + 1] - indptr[b];
            for (int h = 0; h < H; ++h) {
                for (int r = 0; r < cluster_c; ++r) {
                    pieces.push_back({b, h, static_cast<int>(static_cast<int64_t>(P) * r / cluster_c),
                                      static_cast<int>(static_cast<int64_t>(P) * (r + 1) / cluster_c)});
                    cta_of.push_back(static_cast<int>(cta_of.size()));
                }
            }
        }
        grid = static_cast<int>(cta_of.size());
    }
    if (cluster_c > 0) {
        // the cluster pieces are laid out above
    } else if (d.force_splits == 0 && d.max_splits == 0 && !whole_streams) {
        // Balanced line partition: walk the concatenated streams and give each
        // CTA, when it starts, the average of what remains (tokens plus the
        // start-up cost of the pieces still to come), cutting streams at page
        // boundaries. A CTA whose remaining room cannot hold a piece's
        // start-up and half a stage passes the next piece on.
        int64_t streamed = 0, live_streams = 0;
        for (int b = 0; b < B; ++b) {
            streamed += stream_tokens(b);
            if (stream_tokens(b) > 0) live_streams += H;
        }
        const double T0 = static_cast<double>(streamed) * H;
        const double unit_ovh = unit_overhead_tokens(variant);
        const int64_t min_tokens = static_cast<int64_t>(pps) * ps;
        // At least a stage of tokens a CTA, but at least one CTA a stream while
        // they last: a stream costs a unit's start-up wherever it runs, so short
        // streams stacked on few CTAs would queue behind one another.
        grid = static_cast<int>(std::max<int64_t>(
            1, std::min<int64_t>(resident, std::max<int64_t>(static_cast<int64_t>(T0 / min_tokens),
                                                             live_streams))));
        double done = 0.0;                      // tokens assigned so far
        int64_t streams_left = static_cast<int64_t>(B) * H;
        auto budget_for = [&](int c) {
            const double rest =
                (T0 - done) + unit_ovh * static_cast<double>(streams_left + grid - c - 1);
            return rest / (grid - c);
        };
        int c = 0;
        double budget = budget_for(0), used = 0.0;
        for (int b = 0; b < B; ++b) {
            const int P = indptr[b + 1] - indptr[b];
            for (int h = 0; h < H; ++h) {
                int p = start_page[b];
                while (p < P) {
                    if (c < grid - 1 && budget - used - unit_ovh < 0.5 * min_tokens) {
                        ++c;
                        budget = budget_for(c);
                        used = 0.0;
                    }
                    used += unit_ovh;  // the piece's start-up
                    int k = P;
                    const double rest = static_cast<double>(tokens_to(b, P) - tokens_to(b, p));
                    const double room = budget - used;
                    if (c < grid - 1 && room < rest - 0.5 * ps) {
                        k = p + std::max(1, static_cast<int>(std::llround(room / ps)));
                        if (k >= P) k = P;
                    }
                    pieces.push_back({b, h, p, k});
                    cta_of.push_back(c);
                    const double dt = static_cast<double>(tokens_to(b, k) - tokens_to(b, p));
                    used += dt;
                    done += dt;
                    p = k;
                }
                --streams_left;
            }
        }
        grid = cta_of.empty() ? 1 : cta_of.back() + 1;
    } else {
        // Whole streams, or fixed splitting (force_splits, or at most max_splits pieces per
        // stream, 1 = never split): equal pieces, assigned longest first to
        // the least-loaded CTA.
        for (int b = 0; b < B; ++b) {
            const int P0 = start_page[b];
            const int P = indptr[b + 1] - indptr[b] - P0;  // pages the decode kernel streams
            if (P <= 0) continue;
            int n = 1;
            if (whole_streams) {
                n = 1;
            } else if (d.force_splits > 0) {
                n = std::min(d.force_splits, P);
            } else if (d.max_splits > 1) {
                const double T = static_cast<double>(total_tokens) * H;
                const double share_pages = T / static_cast<double>(resident) / ps;
                n = static_cast<int>(std::ceil(P / std::max(1.0, share_pages)));
                n = std::max(1, std::min({n, d.max_splits, P}));
            }
            for (int h = 0; h < H; ++h)
                for (int c = 0; c < n; ++c)
                    pieces.push_back({b, h, P0 + static_cast<int>(static_cast<int64_t>(P) * c / n),
                                      P0 + static_cast<int>(static_cast<int64_t>(P) * (c + 1) / n)});
        }
        grid = static_cast<int>(std::min<int64_t>(resident, static_cast<int64_t>(pieces.size())));
        std::vector<int> order(pieces.size());
        for (size_t i = 0; i < order.size(); ++i) order[i] = static_cast<int>(i);
        auto cost = [&](const Piece& x) { return tokens_to(x.b, x.p1) - tokens_to(x.b, x.p0); };
        std::stable_sort(order.begin(), order.end(),
                         [&](int a, int x) { return cost(pieces[a]) > cost(pieces[x]); });
        std::vector<std::pair<int64_t, int>> heap;  // (load, cta), min-heap
        for (int c = 0; c < grid; ++c) heap.push_back({0, c});
        std::vector<int> assigned(pieces.size(), 0);
        for (int i : order) {
            std::pop_heap(heap.begin(), heap.end(), std::greater<std::pair<int64_t, int>>());
            heap.back().first += cost(pieces[i]) + 64;  // + a stage of per-unit overhead
            assigned[i] = heap.back().second;
            std::push_heap(heap.begin(), heap.end(), std::greater<std::pair<int64_t, int>>());
        }
        std::vector<int> by_cta(order.size());
        for (size_t i = 0; i < by_cta.size(); ++i) by_cta[i] = static_cast<int>(i);
        std::stable_sort(by_cta.begin(), by_cta.end(),
                         [&](int a, int x) { return assigned[a] < assigned[x]; });
        std::vector<Piece> sorted;
        for (int i : by_cta) {
            sorted.push_back(pieces[i]);
            cta_of.push_back(assigned[i]);
        }
        pieces.swap(sorted);
    }
    // Slots for split streams (consecutive per stream) and the merge entries.
    // A cascade plan gives every stream a block of K slots, slot (h*B + b)*K
    // + i: i = 0 holds the prefix state of a cascade request, its suffix
    // pieces (or a split plain stream's pieces) follow, so each merge entry
    // and each prefix tile (requests b0.., stride K) addresses its states
    // contiguously as the kernels expect.
    const int n_pieces = static_cast<int>(pieces.size());
    std::vector<int> slot(pieces.size(), -1);
    std::vector<int4> split_tab;
    int n_slots = 0, max_chunks = 1, casc_K = 0;
    {
        std::vector<std::vector<int>> of_stream(static_cast<size_t>(B) * H);
        for (int i = 0; i < n_pieces; ++i)
            of_stream[static_cast<size_t>(pieces[i].b) * H + pieces[i].h].push_back(i);
        if (!chunks.empty()) {
            size_t most = 1;
            for (const auto& v : of_stream) most = std::max(most, v.size());
            casc_K = static_cast<int>(most) + 1;
            if (static_cast<int64_t>(B) * H * casc_K * G >= (int64_t{1} << 31))
                return OXD_ERR_UNSUPPORTED;
        }
        if (cluster_c > 0) {
            for (int i = 0; i < n_pieces; ++i) slot[i] = i;  // piece r of stream k: k * C + r
            n_slots = n_pieces;
            max_chunks = cluster_c;
        }
        for (size_t st = 0; st < of_stream.size() && cluster_c == 0; ++st) {
            auto& v = of_stream[st];
            max_chunks = std::max(max_chunks, static_cast<int>(v.size()));
            const int b = static_cast<int>(st / H), h = static_cast<int>(st % H);
            const bool casc = start_page[b] > 0;
            if (v.size() < 2 && !casc) continue;
            std::sort(v.begin(), v.end(),
                      [&](int a, int x) { return pieces[a].p0 < pieces[x].p0; });
            if (casc_K > 0) {
                const int blk = (h * B + b) * casc_K;
                split_tab.push_back(make_int4(b * d.num_qo_heads + h * G, casc ? blk : blk + 1,
                                              static_cast<int>(v.size()) + (casc ? 1 : 0), 0));
                int k = blk + 1;
                for (int i : v) slot[i] = k++;
            } else {
                split_tab.push_back(make_int4(b * d.num_qo_heads + h * G, n_slots,
                                              static_cast<int>(v.size()), 0));
                for (int i : v) slot[i] = n_slots++;
            }
        }
        if (casc_K > 0) n_slots = B * H * casc_K;
    }
    // Prefix tiles of a cascade plan (the prefill kernel's work units): the
    // chunk's requests as query "tokens" of q [B][Hq][128], every row seeing
    // the whole prefix (position prefix - 1 for the first), read from the
    // block table of the chunk's first request.
    std::vector<PrefillUnit> punits;
    int64_t shared_kv = 0;
    for (const Chunk& c : chunks) {
        const int64_t L0 =
            static_cast<int64_t>(indptr[c.b0 + 1] - indptr[c.b0] - 1) * ps + last[c.b0];
        int members = 0;
        for (int b = c.b0; b < c.b0 + c.n; ++b) members += start_page[b] > 0 ? 1 : 0;
        shared_kv += static_cast<int64_t>(members - 1) * d.shared_prefix_tokens;
        for (int h = 0; h < H; ++h) {
            PrefillUnit u{};
            u.idx_begin = indptr[c.b0];
            u.n_pages = prefix_pages;
            u.kv_begin = 0;
            u.kv_valid = d.shared_prefix_tokens;
            u.q_begin = c.b0;
            u.n_tok = c.n;
            u.p0 = d.shared_prefix_tokens - 1;
            u.hkv = h;
            u.b = c.b0;
            u.state = (h * B + c.b0) * casc_K;
            u.n_pieces = casc_K;
            u.piece = 0;
            u.qo_b = 0;
            u.kv_len = static_cast<int32_t>(L0);
            u.page_base = indptr[c.b0];
            punits.push_back(u);
        }
    }
    const int n_split = static_cast<int>(split_tab.size());
    // Units: each piece once per 16-row half, on CTAs copies*c + half.
    const int n_units = n_pieces * copies;
    grid *= copies;
    std::vector<int4> units;
    std::vector<int32_t> cta_begin(static_cast<size_t>(grid) + 1, 0);
    {
        std::vector<std::vector<int4>> per_cta(static_cast<size_t>(grid));
        for (int i = 0; i < n_pieces; ++i) {
            const Piece& x = pieces[i];
            const int P = indptr[x.b + 1] - indptr[x.b];
            if (x.p1 - x.p0 >= (1 << kUnitPagesBits)) return OXD_ERR_UNSUPPORTED;
            uint32_t y = static_cast<uint32_t>(x.p1 - x.p0);
            if (x.p1 == P) y |= static_cast<uint32_t>(last[x.b]) << kUnitPagesBits;
            if (x.p0 == 0) y |= 1u << 31;
            for (int half = 0; half < copies; ++half)
                per_cta[static_cast<size_t>(cta_of[i]) * copies + half].push_back(
                    make_int4(indptr[x.b] + x.p0, static_cast<int>(y),
                              x.b | (half << kUnitBBits) | (x.h << (kUnitBBits + 1)), slot[i]));
        }
        for (int c = 0; c < grid; ++c) {
            cta_begin[c] = static_cast<int32_t>(units.size());
            units.insert(units.end(), per_cta[c].begin(), per_cta[c].end());
        }
        cta_begin[grid] = static_cast<int32_t>(units.size());
    }

    // ---- plan object and workspace layout
    oxd_plan P = new (std::nothrow) oxd_plan_s();
    if (P == nullptr) return OXD_ERR_NO_MEMORY;
    P->desc = d;
    P->device = plan_device;
    P->group = G;
    P->variant = variant;
    P->n_items = n_units;
    P->n_slots = n_slots;
    P->n_split = n_split;
    P->max_chunks = max_chunks;
    P->chunk_pages = static_cast<int>(
        std::llround(static_cast<double>(total_tokens) * H * copies / grid / ps));
    P->ctas_per_sm = ctas_per_sm;
    P->num_sms = num_sms;
    P->grid = grid;
    // the prefix tiles of a cascade plan live in the workspace, so a
    // cascade plan's unbound runs upload the whole list
    P->upload = n_units > WorkList::kUnits || grid > WorkList::kCtas ||
                n_split > SplitList::kEntries || !punits.empty();
    P->casc_units = static_cast<int>(punits.size());
    P->cluster_c = cluster_c;
    P->casc_requests = casc_requests;
    P->casc_tile_tokens = kNarrowRows / G;
    P->shared_kv = shared_kv;
    P->nnz = indptr[B];
    P->total_tokens = total_tokens;
    P->off_units = sizeof(WsHeader);
    P->off_cta = align_up(P->off_units + 16 * static_cast<size_t>(n_units), 256);
    P->off_split = align_up(P->off_cta + 32 * static_cast<size_t>(grid), 256);
    P->off_punits = align_up(P->off_split + 16 * std::max<size_t>(split_tab.size(), 1), 256);
    P->meta_bytes = align_up(P->off_punits + sizeof(PrefillUnit) * punits.size(), 256);
    P->off_part_o = P->meta_bytes;
    P->off_part_lse =
        align_up(P->off_part_o + static_cast<size_t>(n_slots) * G * kHeadDim * 4, 256);
    P->ws_bytes = align_up(P->off_part_lse + static_cast<size_t>(n_slots) * G * 4, 256);

    P->work = new (std::nothrow) WorkList();
    P->splits = new (std::nothrow) SplitList();
    P->meta = nullptr;
    P->pinned = false;
    if (P->work == nullptr || P->splits == nullptr) {
        delete P->work;
        delete P->splits;
        delete P;
        return OXD_ERR_NO_MEMORY;
    }
    if (!P->upload) {
        std::copy(units.begin(), units.end(), P->work->unit);
        std::copy(cta_begin.begin(), cta_begin.end(), P->work->cta_begin);
        std::copy(split_tab.begin(), split_tab.end(), P->splits->entry);
    }
    // Workspace image of the list (header stamp 0), for uploads and binds.
    // Lists too long for the parameter buffers are uploaded by every unbound
    // run, so their image is page-locked.
    const size_t image_bytes = P->meta_bytes + 256;
    if (P->upload) {
        P->pinned = cudaHostAlloc(&P->meta, image_bytes, cudaHostAllocDefault) == cudaSuccess;
        if (!P->pinned) cudaGetLastError();  // a host-only plan on a machine without a GPU
    }
    if (P->meta == nullptr) P->meta = std::malloc(image_bytes);
    if (P->meta == nullptr) {
        delete P->work;
        delete P->splits;
        delete P;
        return OXD_ERR_NO_MEMORY;
    }
    {
        uint8_t* m = static_cast<uint8_t*>(P->meta);
        std::memset(m, 0, image_bytes);
        std::memcpy(m + P->off_units, units.data(), 16 * units.size());
        int4* rec = reinterpret_cast<int4*>(m + P->off_cta);
        for (int c = 0; c < grid; ++c) {
            rec[2 * c] = make_int4(cta_begin[c], cta_begin[c + 1], 0, 0);
            rec[2 * c + 1] = cta_begin[c] < cta_begin[c + 1] ? units[cta_begin[c]]
                                                              : make_int4(0, 0, 0, 0);
        }
        std::memcpy(m + P->off_split, split_tab.data(), 16 * split_tab.size());
        if (!punits.empty())
            std::memcpy(m + P->off_punits, punits.data(), sizeof(PrefillUnit) * punits.size());
        P->stamp = next_stamp();
        std::memcpy(m + P->meta_bytes, &P->stamp, sizeof(P->stamp));
    }
    P->bound_ws.store(nullptr);
    P->ev_before = nullptr;
    P->ev_after = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_plans_mu);
        g_plans.insert(P);
    }
    *plan_out = P;
    *ws_out = P->ws_bytes;
    return OXD_OK;
}

oxd_status oxd_plan_get_info(oxd_plan plan, oxd_plan_info* info) {
    if (info == nullptr) return OXD_ERR_INVALID_ARGUMENT;
    if (plan == nullptr || !plan_alive(plan)) return OXD_ERR_PLAN_MISMATCH;
    oxd_plan_info r{};
    r.num_work_items = plan->n_items;
    r.num_split_requests = plan->n_split;
    r.max_chunks = plan->max_chunks;
    r.chunk_pages = plan->chunk_pages;
    r.num_slots = plan->n_slots;
    r.kernel_variant = plan->variant;
    r.grid_ctas = plan->grid;
    r.ctas_per_sm = plan->ctas_per_sm;
    r.num_sms = plan->num_sms;
    r.launches_per_run = plan->n_split > 0 ? 2 : 1;
    r.workspace_bytes = static_cast<int64_t>(plan->ws_bytes);
    r.upload_bytes =
        plan->upload ? static_cast<int64_t>(plan->meta_bytes - plan->off_units) : 0;
    r.total_kv_tokens = plan->total_tokens;
    r.cascade_units = plan->casc_units;
    r.cascade_requests = plan->casc_requests;
    r.shared_kv_tokens = plan->shared_kv;
    r.cluster_size = plan->cluster_c;
    if (plan->cluster_c > 0) r.num_split_requests = plan->n_slots / plan->cluster_c;
    if (plan->casc_units > 0) r.launches_per_run = 3;
    *info = r;
    return OXD_OK;
}

oxd_status oxd_plan_set_timing_events(oxd_plan plan, void* before, void* after) {
    if (plan == nullptr || !plan_alive(plan)) return OXD_ERR_PLAN_MISMATCH;
    if ((before == nullptr) != (after == nullptr)) return OXD_ERR_INVALID_ARGUMENT;
    plan->ev_before = static_cast<cudaEvent_t>(before);
    plan->ev_after = static_cast<cudaEvent_t>(after);
    return OXD_OK;
}

oxd_status oxd_plan_bind_workspace(oxd_plan plan, void* workspace, size_t workspace_bytes,
                                   void* stream) {
    if (plan == nullptr || !plan_alive(plan)) return OXD_ERR_PLAN_MISMATCH;
    if (workspace == nullptr) return OXD_ERR_INVALID_ARGUMENT;
    if (!aligned(workspace, 256)) return OXD_ERR_ALIGNMENT;
    if (workspace_bytes < plan->ws_bytes) return OXD_ERR_WORKSPACE_TOO_SMALL;
    if (plan->device < 0) return OXD_ERR_PLAN_MISMATCH;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) return OXD_ERR_CUDA;
    if (cur != plan->device) return OXD_ERR_PLAN_MISMATCH;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const uint8_t* m = static_cast<const uint8_t*>(plan->meta);
    // The list first, then the stamp that makes it valid.
    if (cudaMemcpyAsync(ws + plan->off_units, m + plan->off_units,
                        plan->meta_bytes - plan->off_units, cudaMemcpyHostToDevice,
                        s) != cudaSuccess ||
        cudaMemcpyAsync(ws + offsetof(WsHeader, stamp), m + plan->meta_bytes,
                        sizeof(unsigned long long), cudaMemcpyHostToDevice, s) != cudaSuccess)
        return OXD_ERR_CUDA;
    plan->bound_ws.store(workspace);
    return OXD_OK;
}

oxd_status oxd_plan_destroy(oxd_plan plan) {
    if (plan == nullptr) return OXD_ERR_INVALID_ARGUMENT;
    {
        std::lock_guard<std::mutex> lk(g_plans_mu);
        if (g_plans.erase(plan) == 0) return OXD_ERR_PLAN_MISMATCH;
    }
    if (plan->pinned)
        cudaFreeHost(plan->meta);
    else
        std::free(plan->meta);
    delete plan->work;
    delete plan->splits;
    delete plan;
    return OXD_OK;
}

oxd_status oxd_paged_decode_run(oxd_plan plan, const void* q, const void* k_pages,
                                const void* v_pages, const int32_t* indptr,
                                const int32_t* indices, const int32_t* last_page_len,
                                float sm_scale, void* out, float* lse, void* workspace,
                                size_t workspace_bytes, void* stream) {
    if (plan == nullptr || !plan_alive(plan)) return OXD_ERR_PLAN_MISMATCH;
    if (q == nullptr || k_pages == nullptr || v_pages == nullptr || indptr == nullptr ||
        indices == nullptr || last_page_len == nullptr || out == nullptr || workspace == nullptr)
        return OXD_ERR_INVALID_ARGUMENT;
    if (!std::isfinite(sm_scale)) return OXD_ERR_INVALID_ARGUMENT;
    const oxd_paged_decode_desc& d = plan->desc;
    if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(out, 16) ||
        !aligned(indptr, 4) || !aligned(indices, 4) || !aligned(last_page_len, 4) ||
        !aligned(lse, 4) || !aligned(workspace, 256))
        return OXD_ERR_ALIGNMENT;
    if (workspace_bytes < plan->ws_bytes) return OXD_ERR_WORKSPACE_TOO_SMALL;

    const size_t rows = static_cast<size_t>(d.batch) * d.num_qo_heads;
    const size_t pool = static_cast<size_t>(d.num_pages) * d.page_size * d.num_kv_heads *
                        d.head_dim * 2;
    const Span in[] = {span(q, rows * kHeadDim * 2),
                       span(k_pages, pool),
                       span(v_pages, pool),
                       span(indptr, (static_cast<size_t>(d.batch) + 1) * 4),
                       span(indices, static_cast<size_t>(plan->nnz) * 4),
                       span(last_page_len, static_cast<size_t>(d.batch) * 4)};
    const Span outs[] = {span(out, rows * kHeadDim * 2),
                         lse ? span(lse, rows * 4) : Span{0, 0},
                         span(workspace, plan->ws_bytes)};
    for (const Span& o : outs) {
        for (const Span& i : in)
            if (overlap(o, i)) return OXD_ERR_ALIAS;
    }
    if (overlap(outs[0], outs[1]) || overlap(outs[0], outs[2]) || overlap(outs[1], outs[2]))
        return OXD_ERR_ALIAS;

    if (plan->device >= 0) {
        int cur = -1;
        if (cudaGetDevice(&cur) != cudaSuccess) return OXD_ERR_CUDA;
        if (cur != plan->device) return OXD_ERR_PLAN_MISMATCH;
    }
    CUtensorMap tk, tv, tq, tq3;
    if (!encode_pool(&tk, k_pages, d) || !encode_pool(&tv, v_pages, d)) return OXD_ERR_CUDA;
    if (plan->variant == kVariantWide && !encode_q(&tq, q, d)) return OXD_ERR_CUDA;
    if (plan->casc_units > 0) {
        // q [B][Hq][128] as (d, head, request) for the prefix tiles: a box is
        // 64 columns x the G heads of one KV head x up to 128 / G requests
        const uint64_t dims[3] = {static_cast<uint64_t>(kHeadDim),
                                  static_cast<uint64_t>(d.num_qo_heads),
                                  static_cast<uint64_t>(d.batch)};
        const uint64_t strides[2] = {static_cast<uint64_t>(kHeadDim) * 2,
                                     static_cast<uint64_t>(d.num_qo_heads) * kHeadDim * 2};
        const uint32_t box[3] = {64, static_cast<uint32_t>(plan->group),
                                 static_cast<uint32_t>(plan->casc_tile_tokens)};
        if (!encode_bf16_map(&tq3, q, 3, dims, strides, box)) return OXD_ERR_CUDA;
    }

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const bool bound = plan->bound_ws.load() == workspace;
    // An unbound run with a long list uploads it together with a zero stamp,
    // which also ends any binding of another plan to this workspace.
    const bool in_ws = bound || plan->upload;
    constexpr size_t kStampOff = offsetof(WsHeader, stamp);
    if (!bound && plan->upload &&
        cudaMemcpyAsync(ws + kStampOff, static_cast<uint8_t*>(plan->meta) + kStampOff,
                        plan->meta_bytes - kStampOff, cudaMemcpyHostToDevice,
                        s) != cudaSuccess)
        return OXD_ERR_CUDA;

    DecodeParams p{};
    p.q = static_cast<const uint16_t*>(q);
    p.out = static_cast<uint16_t*>(out);
    p.lse = lse;
    p.indptr = indptr;
    p.indices = indices;
    p.last_page_len = last_page_len;
    p.units = in_ws ? reinterpret_cast<const int4*>(ws + plan->off_units) : nullptr;
    p.cta_rec = in_ws ? reinterpret_cast<const int4*>(ws + plan->off_cta) : nullptr;
    p.ws_stamp = bound ? reinterpret_cast<const unsigned long long*>(ws + kStampOff) : nullptr;
    p.stamp = plan->stamp;
    p.clear_stamp = bound ? nullptr : reinterpret_cast<unsigned long long*>(ws + kStampOff);
    p.n_units = plan->n_items;
    p.n_slots = plan->n_slots;
    p.batch = d.batch;
    p.nnz = plan->nnz;
    p.part_o = reinterpret_cast<float*>(ws + plan->off_part_o);
    p.part_lse = reinterpret_cast<float*>(ws + plan->off_part_lse);
    p.status = reinterpret_cast<unsigned long long*>(ws + offsetof(WsHeader, status));
    p.last_epoch = reinterpret_cast<uint32_t*>(ws + offsetof(WsHeader, last_epoch));
    p.epoch = next_epoch();
    p.num_qo_heads = d.num_qo_heads;
    p.num_kv_heads = d.num_kv_heads;
    p.group = plan->group;
    p.page_size = d.page_size;
    p.layout = d.layout;
    p.num_pages = d.num_pages;
    p.scale_log2 = sm_scale * 1.4426950408889634f;  // log2(e)
    p.cluster_c = plan->cluster_c;
    p.wait_ns = d.wait_timeout_ns > 0 ? d.wait_timeout_ns : kWaitTimeoutNs;

    if (plan->ev_before != nullptr && cudaEventRecord(plan->ev_before, s) != cudaSuccess)
        return OXD_ERR_CUDA;
    const WorkList* inline_list = in_ws ? nullptr : plan->work;
    // A programmatic dependent launch only where the decode kernel directly
    // follows the caller's previous work on the stream (no copy or timing
    // event of this run in between).
    const bool pdl = d.pdl != 0 && plan->ev_before == nullptr && !(!bound && plan->upload);
    const cudaError_t le =
        plan->variant == kVariantWide
            ? launch_decode_wide(tk, tv, tq, p, inline_list, plan->grid, s, pdl)
            : launch_decode(plan->variant, tk, tv, p, inline_list, plan->grid, s, pdl);
    if (le != cudaSuccess) return OXD_ERR_CUDA;
    if (plan->ev_after != nullptr && cudaEventRecord(plan->ev_after, s) != cudaSuccess)
        return OXD_ERR_CUDA;
    if (plan->casc_units > 0) {
        // the shared prefixes: every prefix tile writes slot i = 0 of its
        // requests' streams (the decode kernel writes the others). Launched
        // early behind the decode kernel, its CTAs fill the SMs the decode
        // CTAs leave; each waits for the decode grid before it exits, so the
        // merge, which waits for this grid, sees both kernels' states.
        PrefillParams pp{};
        pp.q = p.q;
        pp.indptr = indptr;
        pp.indices = indices;
        pp.last_page_len = last_page_len;
        pp.qo_indptr = nullptr;  // the query rows are the batch's own
        pp.units = reinterpret_cast<const PrefillUnit*>(ws + plan->off_punits);
        pp.ws_stamp = p.ws_stamp;
        pp.stamp = p.stamp;
        pp.clear_stamp = nullptr;
        pp.part_o = p.part_o;
        pp.part_lse = p.part_lse;
        pp.n_states = static_cast<int64_t>(plan->n_slots) * plan->group;
        pp.status = p.status;
        pp.last_epoch = p.last_epoch;
        pp.epoch = p.epoch;
        pp.n_units = plan->casc_units;
        pp.batch = d.batch;
        pp.n_q_tokens = d.batch;
        pp.nnz = plan->nnz;
        pp.num_qo_heads = d.num_qo_heads;
        pp.num_kv_heads = d.num_kv_heads;
        pp.group = plan->group;
        pp.tile_tokens = plan->casc_tile_tokens;
        pp.page_size = d.page_size;
        pp.layout = d.layout;
        pp.num_pages = d.num_pages;
        pp.scale_log2 = p.scale_log2;
        pp.wait_prior = 1;
        pp.wait_ns = p.wait_ns;
        if (launch_prefill_narrow(tk, tv, tq3, pp, plan->casc_units, s,
                                  plan->ev_after == nullptr) != cudaSuccess)
            return OXD_ERR_CUDA;
    }
    if (plan->n_split > 0) {
        MergeParams mp{};
        mp.v = p.part_o;
        mp.s = p.part_lse;
        mp.out = p.out;
        mp.lse = lse;
        mp.entries = in_ws ? reinterpret_cast<const int4*>(ws + plan->off_split) : nullptr;
        mp.ws_stamp = p.ws_stamp;
        mp.stamp = p.stamp;
        mp.n_rows = static_cast<int64_t>(d.batch) * d.num_qo_heads;
        mp.n_states = static_cast<int64_t>(plan->n_slots) * plan->group;
        mp.uniform = 0;
        mp.n = plan->n_split;
        mp.S = 0;
        mp.R = plan->group;
        mp.D = kHeadDim;
        mp.s_to_ln = 0.693147180559945309f;  // partial LSEs are log2
        mp.max_count = plan->max_chunks + (plan->casc_units > 0 ? 1 : 0);
        // With timing events the decode kernel must end before ev_after, so
        // the merge is then launched without the early-start attribute.
        if (launch_split_merge(mp, in_ws ? nullptr : plan->splits, s,
                               plan->ev_after == nullptr) != cudaSuccess)
            return OXD_ERR_CUDA;
    }
    return OXD_OK;
}

oxd_status oxd_merge_states(const float* v, const float* s, int32_t N, int32_t S, int32_t H,
                            int32_t D, void* v_out, float* s_out, void* stream) {
    if (v == nullptr || s == nullptr || v_out == nullptr) return OXD_ERR_INVALID_ARGUMENT;
    if (N < 1 || S < 1 || H < 1 || D < 4 || D % 4 != 0) return OXD_ERR_INVALID_ARGUMENT;
    if (!aligned(v, 16) || !aligned(s, 4) || !aligned(v_out, 8) || !aligned(s_out, 4))
        return OXD_ERR_ALIGNMENT;
    const size_t NH = static_cast<size_t>(N) * H;
    const Span in[] = {span(v, NH * S * D * 4), span(s, NH * S * 4)};
    const Span outs[] = {span(v_out, NH * D * 2), s_out ? span(s_out, NH * 4) : Span{0, 0}};
    for (const Span& o : outs)
        for (const Span& i : in)
            if (overlap(o, i)) return OXD_ERR_ALIAS;
    if (overlap(outs[0], outs[1])) return OXD_ERR_ALIAS;
    MergeParams mp{};
    mp.v = v;
    mp.s = s;
    mp.out = static_cast<uint16_t*>(v_out);
    mp.lse = s_out;
    mp.entries = nullptr;
    mp.uniform = 1;
    mp.n = N;
    mp.S = S;
    mp.R = H;
    mp.D = D;
    mp.s_to_ln = 1.0f;
    mp.max_count = S;
    if (launch_merge(mp, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return OXD_ERR_CUDA;
    return OXD_OK;
}

oxd_status oxd_read_device_status(const void* workspace, void* stream, int32_t* code) {
    if (workspace == nullptr || code == nullptr) return OXD_ERR_INVALID_ARGUMENT;
    if (!aligned(workspace, 256)) return OXD_ERR_ALIGNMENT;
    WsHeader h;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&h, workspace, 16, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return OXD_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return OXD_ERR_CUDA;
    // A code counts only if the last run that started recorded it.
    const int32_t c = static_cast<uint32_t>(h.status >> 32) == h.last_epoch
                          ? static_cast<int32_t>(static_cast<uint32_t>(h.status))
                          : OXD_DEVICE_OK;
    *code = c;
    return c == OXD_DEVICE_OK ? OXD_OK : OXD_ERR_DEVICE_STATUS;
}

}  // extern "C"

extern "C" oxd_status oxd_rope_append(const oxd_rope_append_desc* desc, const void* q,
                                      const void* k, const void* v,
                                      const int32_t* token_request, const int32_t* positions,
                                      const int32_t* indptr, const int32_t* indices,
                                      const int32_t* page_refcount, void* q_out, void* k_pages,
                                      void* v_pages, void* workspace, size_t workspace_bytes,
                                      void* stream) {
    if (desc == nullptr || q == nullptr || k == nullptr || v == nullptr ||
        token_request == nullptr || positions == nullptr || indptr == nullptr ||
        indices == nullptr || page_refcount == nullptr || q_out == nullptr ||
        k_pages == nullptr || v_pages == nullptr || workspace == nullptr)
        return OXD_ERR_INVALID_ARGUMENT;
    const oxd_rope_append_desc& d = *desc;
    if (d.num_tokens < 1 || d.batch < 1 || d.num_qo_heads < 1 || d.num_kv_heads < 1 ||
        d.num_pages < 1 || d.num_indices < 1 || d.reserved[0] != 0 || d.reserved[1] != 0 ||
        (d.layout != OXD_LAYOUT_NHD && d.layout != OXD_LAYOUT_HND) ||
        !(std::isfinite(d.rope_theta) && d.rope_theta > 1.0))
        return OXD_ERR_INVALID_ARGUMENT;
    if (d.head_dim != kHeadDim) return OXD_ERR_UNSUPPORTED;
    if (d.page_size != 8 && d.page_size != 16 && d.page_size != 32 && d.page_size != 64)
        return OXD_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(d.num_tokens) * (d.num_qo_heads + d.num_kv_heads) >
        (int64_t{1} << 33))
        return OXD_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(q_out, 16) ||
        !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(token_request, 4) ||
        !aligned(positions, 4) || !aligned(indptr, 4) || !aligned(indices, 4) ||
        !aligned(page_refcount, 4) || !aligned(workspace, 256))
        return OXD_ERR_ALIGNMENT;
    if (workspace_bytes < sizeof(WsHeader)) return OXD_ERR_WORKSPACE_TOO_SMALL;
    const size_t T = static_cast<size_t>(d.num_tokens);
    const size_t qbytes = T * d.num_qo_heads * kHeadDim * 2;
    const size_t kvbytes = T * d.num_kv_heads * kHeadDim * 2;
    const size_t pool = static_cast<size_t>(d.num_pages) * d.page_size * d.num_kv_heads *
                        kHeadDim * 2;
    const Span in[] = {span(k, kvbytes), span(v, kvbytes), span(token_request, T * 4),
                       span(positions, T * 4),
                       span(indptr, (static_cast<size_t>(d.batch) + 1) * 4),
                       span(indices, static_cast<size_t>(d.num_indices) * 4),
                       span(page_refcount, static_cast<size_t>(d.num_pages) * 4)};
    const Span qin = span(q, qbytes);
    const Span outs[] = {span(q_out, qbytes), span(k_pages, pool), span(v_pages, pool),
                         span(workspace, sizeof(WsHeader))};
    for (const Span& o : outs) {
        for (const Span& i : in)
            if (overlap(o, i)) return OXD_ERR_ALIAS;
    }
    // q_out may be q exactly (each row is read before it is written, by the
    // same warp); any other overlap with q is refused
    if (q_out != q && overlap(outs[0], qin)) return OXD_ERR_ALIAS;
    for (int i = 1; i < 4; ++i)
        if (overlap(outs[i], qin)) return OXD_ERR_ALIAS;
    for (int i = 0; i < 4; ++i)
        for (int j = i + 1; j < 4; ++j)
            if (overlap(outs[i], outs[j])) return OXD_ERR_ALIAS;

    AppendParams p{};
    p.q = static_cast<const uint16_t*>(q);
    p.k = static_cast<const uint16_t*>(k);
    p.v = static_cast<const uint16_t*>(v);
    p.token_request = token_request;
    p.positions = positions;
    p.indptr = indptr;
    p.indices = indices;
    p.refcount = page_refcount;
    p.q_out = static_cast<uint16_t*>(q_out);
    p.k_pages = static_cast<uint16_t*>(k_pages);
    p.v_pages = static_cast<uint16_t*>(v_pages);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.status = reinterpret_cast<unsigned long long*>(ws + offsetof(WsHeader, status));
    p.last_epoch = reinterpret_cast<uint32_t*>(ws + offsetof(WsHeader, last_epoch));
    p.epoch = next_run_epoch();
    p.T = d.num_tokens;
    p.B = d.batch;
    p.Hq = d.num_qo_heads;
    p.Hkv = d.num_kv_heads;
    p.page_size = d.page_size;
    p.layout = d.layout;
    p.num_indices = d.num_indices;
    p.num_pages = d.num_pages;
    for (int i = 0; i < kHeadDim / 2; ++i) {
        // frequency in turns per position, f / (2 pi), split into two floats
        const double g = std::pow(d.rope_theta, -2.0 * static_cast<double>(i) / kHeadDim) /
                         6.283185307179586476925286766559;
        p.turns_hi[i] = static_cast<float>(g);
        p.turns_lo[i] = static_cast<float>(g - static_cast<double>(p.turns_hi[i]));
    }
    if (launch_rope_append(p, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return OXD_ERR_CUDA;
    return OXD_OK;
}
