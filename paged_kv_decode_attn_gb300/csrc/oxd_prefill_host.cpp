// Host side of the paged causal prefill: planning, operand checks, enqueue.
//
// "FlashInfer parity matrix" page, "Admitted attention matrix", row "Paged
// causal prefill" (caller-owned F32 workspace for the split pieces), driven
// as the "Oxide Infer" README's "One execution model" describes: the plan
// picks the tile size (256 rows on the two-half kernel, or 128 rows on the
// narrow kernel for prefills too short to fill the GPU with the former) and
// fixes the tiles, the pieces of long tiles and the workspace; a run checks
// operands and enqueues (the work list copied into the workspace first,
// unless the workspace is bound to the plan), the prefill kernel and, when
// some tile was split, the merge kernel behind it.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <limits>
#include <mutex>
#include <new>
#include <unordered_set>
#include <vector>

#include "../../include/oxd.h"
#include "oxd_host_util.h"
#include "oxd_internal.h"
#include "oxd_prefill.h"

using namespace oxd;

struct oxd_prefill_plan_s {
    oxd_paged_prefill_desc desc;
    int device;  // -1: host-only plan
    int group;
    bool narrow;  // 128-row tiles on the narrow kernel, else 256-row tiles
    int tile_tokens;
    int n_tiles;
    int n_units;
    int n_split_tiles;
    int max_pieces;
    int n_entries;
    int ctas_per_sm;
    int num_sms;
    int64_t n_groups;  // partial-state groups (G rows each)
    int64_t nq;
    int64_t nnz;
    int64_t total_kv;
    int64_t pairs;
    size_t off_units, off_entries, meta_bytes, off_part_o, off_part_lse, ws_bytes;
    void* meta;  // workspace image [0, meta_bytes) (stamp word 0), then the plan's stamp
    bool pinned;
    unsigned long long stamp;
    std::atomic<const void*> bound_ws;
    cudaEvent_t ev_before, ev_after;
};

namespace {

// a piece streams at least 128 cached tokens: one stage of the two-half
// kernel, two of the narrow one
constexpr int kMinPieceTokens = 128;
constexpr int kMaxPieces = 64;

std::mutex g_mu;
std::unordered_set<oxd_prefill_plan> g_live;

bool alive(oxd_prefill_plan p) {
    std::lock_guard<std::mutex> lk(g_mu);
    return g_live.count(p) != 0;
}

oxd_status check_desc(const oxd_paged_prefill_desc& d) {
    if (d.batch < 1 || d.num_qo_heads < 1 || d.num_kv_heads < 1 || d.head_dim < 1 ||
        d.page_size < 1 || d.num_pages < 1 || d.max_splits < 0 || d.num_sms < 0)
        return OXD_ERR_INVALID_ARGUMENT;
    if (d.num_qo_heads % d.num_kv_heads != 0) return OXD_ERR_INVALID_ARGUMENT;
    if (d.layout != OXD_LAYOUT_NHD && d.layout != OXD_LAYOUT_HND) return OXD_ERR_INVALID_ARGUMENT;
    if (d.wait_timeout_ns < 0) return OXD_ERR_INVALID_ARGUMENT;
    if ((d.tile_rows != 0 && d.tile_rows != kNarrowRows && d.tile_rows != kPrefillRows) ||
        d.reserved != 0)
        return OXD_ERR_INVALID_ARGUMENT;
    if (d.head_dim != kHeadDim) return OXD_ERR_UNSUPPORTED;
    if (d.page_size != 8 && d.page_size != 16 && d.page_size != 32 && d.page_size != 64)
        return OXD_ERR_UNSUPPORTED;
    if (d.num_qo_heads / d.num_kv_heads > kMaxPrefillGroup) return OXD_ERR_UNSUPPORTED;
    if (d.num_pages >= (int64_t{1} << 31)) return OXD_ERR_UNSUPPORTED;
    return OXD_OK;
}

void free_plan(oxd_prefill_plan P) {
    if (P->pinned)
        cudaFreeHost(P->meta);
    else
        std::free(P->meta);
    delete P;
}

}  // namespace

extern "C" {

oxd_status oxd_paged_prefill_plan(const oxd_paged_prefill_desc* desc, const int32_t* qo_indptr,
                                  const int32_t* indptr, const int32_t* last, int device,
                                  oxd_prefill_plan* plan_out, size_t* ws_out) {
    if (desc == nullptr || qo_indptr == nullptr || indptr == nullptr || last == nullptr ||
        plan_out == nullptr || ws_out == nullptr)
        return OXD_ERR_INVALID_ARGUMENT;
    const oxd_paged_prefill_desc d = *desc;
    oxd_status st = check_desc(d);
    if (st != OXD_OK) return st;
    const int B = d.batch, ps = d.page_size, H = d.num_kv_heads;
    const int G = d.num_qo_heads / H;
    if (qo_indptr[0] != 0 || indptr[0] < 0) return OXD_ERR_INVALID_ARGUMENT;
    int64_t total_kv = 0, pairs = 0;
    for (int b = 0; b < B; ++b) {
        const int64_t P = static_cast<int64_t>(indptr[b + 1]) - indptr[b];
        const int64_t q = static_cast<int64_t>(qo_indptr[b + 1]) - qo_indptr[b];
        if (P < 1 || last[b] < 1 || last[b] > ps || q < 0) return OXD_ERR_INVALID_ARGUMENT;
        const int64_t L = (P - 1) * ps + last[b];
        if (q > L) return OXD_ERR_INVALID_ARGUMENT;
        if (L >= (int64_t{1} << 30)) return OXD_ERR_UNSUPPORTED;
        total_kv += L;
        pairs += q * (L - q) + q * (q + 1) / 2;
    }
    const int64_t nq = qo_indptr[B];
    if (nq * d.num_qo_heads >= (int64_t{1} << 31) || static_cast<int64_t>(indptr[B]) < 1)
        return OXD_ERR_UNSUPPORTED;

    int num_sms = d.num_sms, plan_device = -1;
    if (num_sms == 0) {
        if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, device) !=
                cudaSuccess ||
            num_sms < 1)
            return OXD_ERR_CUDA;
        plan_device = device;
    }
    // Stages of tiles of `rows` rows over stages of `stage` tokens (each
    // tile streams its request's cached tokens up to its last query token).
    auto count_stages = [&](int rows, int stage) {
        const int Tr = rows / G;
        int64_t n = 0;
        for (int b = 0; b < B; ++b) {
            const int q_len = qo_indptr[b + 1] - qo_indptr[b];
            const int64_t L = static_cast<int64_t>(indptr[b + 1] - indptr[b] - 1) * ps + last[b];
            for (int qt = 0; qt * Tr < q_len; ++qt) {
                const int64_t kv_end = L - q_len + qt * Tr + std::min(Tr, q_len - qt * Tr);
                n += H * ((kv_end + stage - 1) / stage);
            }
        }
        return n;
    };
    // The two-half kernel needs a whole SM a tile; a prefill that would not
    // give every SM one of its stages runs sooner as smaller tiles, two a SM.
    const bool narrow = d.tile_rows == kNarrowRows ||
                        (d.tile_rows == 0 &&
                         count_stages(kPrefillRows, kPrefillStageTokens) < num_sms);
    const int rows = narrow ? kNarrowRows : kPrefillRows;
    const int stage_tokens = narrow ? kNarrowStageTokens : kPrefillStageTokens;
    const int T = rows / G;
    int ctas_per_sm = 0;
    if (plan_device >= 0) {
        int prev = 0;
        if (cudaGetDevice(&prev) != cudaSuccess) return OXD_ERR_CUDA;
        if (cudaSetDevice(device) != cudaSuccess) return OXD_ERR_CUDA;
        const cudaError_t e =
            narrow ? prefill_narrow_occupancy(&ctas_per_sm) : prefill_occupancy(&ctas_per_sm);
        cudaSetDevice(prev);
        if (e != cudaSuccess) return OXD_ERR_CUDA;
    }
    if (ctas_per_sm < 1) {
        int smem = 0;
        if (narrow)
            prefill_narrow_smem_bytes(&smem);
        else
            prefill_smem_bytes(&smem);
        ctas_per_sm = std::max(1, std::min(2, (228 * 1024) / (smem + 1024)));
    }

    // ---- tiles: up to T query tokens of one request with the G heads of one
    // KV head; a tile streams its request's cached tokens up to the position
    // of its last query token.
    struct Tile {
        int b, hkv, q0, n_tok, p0, stages, kv_end;
    };
    std::vector<Tile> tiles;
    int64_t total_stages = 0;
    for (int b = 0; b < B; ++b) {
        const int q_len = qo_indptr[b + 1] - qo_indptr[b];
        const int64_t L = static_cast<int64_t>(indptr[b + 1] - indptr[b] - 1) * ps + last[b];
        for (int qt = 0; qt * T < q_len; ++qt) {
            const int n_tok = std::min(T, q_len - qt * T);
            const int p0 = static_cast<int>(L - q_len + qt * T);
            const int kv_end = p0 + n_tok;
            const int stages = (kv_end + stage_tokens - 1) / stage_tokens;
            for (int h = 0; h < H; ++h) {
                tiles.push_back({b, h, qo_indptr[b] + qt * T, n_tok, p0, stages, kv_end});
                total_stages += stages;
            }
        }
    }
    if (tiles.empty()) return OXD_ERR_INVALID_ARGUMENT;  // no query token at all
    // ---- pieces: when the tiles alone do not fill the resident CTAs, long
    // tiles are cut into pieces of about equal stage counts
    const int64_t resident = static_cast<int64_t>(num_sms) * ctas_per_sm;
    int64_t chunk = std::numeric_limits<int64_t>::max();
    if (d.max_splits != 1 && static_cast<int64_t>(tiles.size()) < resident)
        chunk = std::max<int64_t>(kMinPieceTokens / stage_tokens,
                                  (total_stages + resident - 1) / resident);
    const int cap = d.max_splits > 1 ? std::min(d.max_splits, kMaxPieces) : kMaxPieces;
    std::vector<PrefillUnit> units;
    std::vector<int4> entries;
    int64_t n_groups = 0;
    int n_split = 0, max_pieces = 1;
    for (const Tile& t : tiles) {
        int S = 1;
        if (chunk != std::numeric_limits<int64_t>::max())
            S = static_cast<int>(std::min<int64_t>(
                {(t.stages + chunk - 1) / chunk, static_cast<int64_t>(cap),
                 static_cast<int64_t>(t.stages)}));
        S = std::max(1, S);
        max_pieces = std::max(max_pieces, S);
        int state = 0;
        if (S > 1) {
            ++n_split;
            if (n_groups + static_cast<int64_t>(t.n_tok) * S >= (int64_t{1} << 31) / rows)
                return OXD_ERR_UNSUPPORTED;
            state = static_cast<int>(n_groups);
            n_groups += static_cast<int64_t>(t.n_tok) * S;
            for (int i = 0; i < t.n_tok; ++i)
                entries.push_back(make_int4((t.q0 + i) * d.num_qo_heads + t.hkv * G,
                                            state + i * S, S, 0));
        }
        const int64_t L = static_cast<int64_t>(indptr[t.b + 1] - indptr[t.b] - 1) * ps + last[t.b];
        for (int i = 0; i < S; ++i) {
            const int s0 = static_cast<int>(static_cast<int64_t>(t.stages) * i / S);
            const int s1 = static_cast<int>(static_cast<int64_t>(t.stages) * (i + 1) / S);
            PrefillUnit u{};
            u.kv_begin = s0 * stage_tokens;
            u.kv_valid = std::min(t.kv_end, s1 * stage_tokens) - u.kv_begin;
            u.idx_begin = indptr[t.b] + u.kv_begin / ps;
            u.n_pages = (u.kv_valid + ps - 1) / ps;
            u.q_begin = t.q0;
            u.n_tok = t.n_tok;
            u.p0 = t.p0;
            u.hkv = t.hkv;
            u.b = t.b;
            u.state = state;
            u.n_pieces = S;
            u.piece = i;
            u.qo_b = qo_indptr[t.b];
            u.kv_len = static_cast<int32_t>(L);
            u.page_base = indptr[t.b];
            units.push_back(u);
        }
    }
    // longest pieces first: the block scheduler starts CTAs in grid order
    std::stable_sort(units.begin(), units.end(), [](const PrefillUnit& a, const PrefillUnit& x) {
        return a.kv_valid > x.kv_valid;
    });
    if (units.size() >= (size_t{1} << 31)) return OXD_ERR_UNSUPPORTED;

    oxd_prefill_plan P = new (std::nothrow) oxd_prefill_plan_s();
    if (P == nullptr) return OXD_ERR_NO_MEMORY;
    P->desc = d;
    P->device = plan_device;
    P->group = G;
    P->narrow = narrow;
    P->tile_tokens = T;
    P->n_tiles = static_cast<int>(tiles.size());
    P->n_units = static_cast<int>(units.size());
    P->n_split_tiles = n_split;
    P->max_pieces = max_pieces;
    P->n_entries = static_cast<int>(entries.size());
    P->ctas_per_sm = ctas_per_sm;
    P->num_sms = num_sms;
    P->n_groups = n_groups;
    P->nq = nq;
    P->nnz = indptr[B];
    P->total_kv = total_kv;
    P->pairs = pairs;
    P->off_units = sizeof(WsHeader);
    P->off_entries = align_up(P->off_units + sizeof(PrefillUnit) * units.size(), 256);
    P->meta_bytes = align_up(P->off_entries + 16 * std::max<size_t>(entries.size(), 1), 256);
    P->off_part_o = P->meta_bytes;
    P->off_part_lse =
        align_up(P->off_part_o + static_cast<size_t>(n_groups) * G * kHeadDim * 4, 256);
    P->ws_bytes = align_up(P->off_part_lse + static_cast<size_t>(n_groups) * G * 4, 256);
    const size_t image_bytes = P->meta_bytes + 256;
    P->pinned = false;
    P->meta = nullptr;
    if (plan_device >= 0) {
        P->pinned = cudaHostAlloc(&P->meta, image_bytes, cudaHostAllocDefault) == cudaSuccess;
        if (!P->pinned) {
            cudaGetLastError();
            P->meta = nullptr;
        }
    }
    if (P->meta == nullptr) P->meta = std::malloc(image_bytes);
    if (P->meta == nullptr) {
        delete P;
        return OXD_ERR_NO_MEMORY;
    }
    {
        uint8_t* m = static_cast<uint8_t*>(P->meta);
        std::memset(m, 0, image_bytes);
        std::memcpy(m + P->off_units, units.data(), sizeof(PrefillUnit) * units.size());
        if (!entries.empty()) std::memcpy(m + P->off_entries, entries.data(), 16 * entries.size());
        P->stamp = next_plan_stamp();
        std::memcpy(m + P->meta_bytes, &P->stamp, sizeof(P->stamp));
    }
    P->bound_ws.store(nullptr);
    P->ev_before = nullptr;
    P->ev_after = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        g_live.insert(P);
    }
    *plan_out = P;
    *ws_out = P->ws_bytes;
    return OXD_OK;
}

oxd_status oxd_prefill_plan_get_info(oxd_prefill_plan plan, oxd_prefill_plan_info* info) {
    if (info == nullptr) return OXD_ERR_INVALID_ARGUMENT;
    if (plan == nullptr || !alive(plan)) return OXD_ERR_PLAN_MISMATCH;
    oxd_prefill_plan_info r{};
    r.tile_tokens = plan->tile_tokens;
    r.num_tiles = plan->n_tiles;
    r.num_units = plan->n_units;
    r.num_split_tiles = plan->n_split_tiles;
    r.max_pieces = plan->max_pieces;
    r.num_merge_rows = plan->n_entries * plan->group;
    r.launches_per_run = plan->n_entries > 0 ? 2 : 1;
    r.ctas_per_sm = plan->ctas_per_sm;
    r.num_sms = plan->num_sms;
    r.tile_rows = plan->narrow ? kNarrowRows : kPrefillRows;
    r.workspace_bytes = static_cast<int64_t>(plan->ws_bytes);
    r.total_q_tokens = plan->nq;
    r.total_kv_tokens = plan->total_kv;
    r.causal_pairs = plan->pairs;
    *info = r;
    return OXD_OK;
}

oxd_status oxd_prefill_plan_set_timing_events(oxd_prefill_plan plan, void* before, void* after) {
    if (plan == nullptr || !alive(plan)) return OXD_ERR_PLAN_MISMATCH;
    if ((before == nullptr) != (after == nullptr)) return OXD_ERR_INVALID_ARGUMENT;
    plan->ev_before = static_cast<cudaEvent_t>(before);
    plan->ev_after = static_cast<cudaEvent_t>(after);
    return OXD_OK;
}

oxd_status oxd_prefill_plan_bind_workspace(oxd_prefill_plan plan, void* workspace,
                                           size_t workspace_bytes, void* stream) {
    if (plan == nullptr || !alive(plan)) return OXD_ERR_PLAN_MISMATCH;
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
    // the list first, then the stamp that makes it valid
    if (cudaMemcpyAsync(ws + plan->off_units, m + plan->off_units,
                        plan->meta_bytes - plan->off_units, cudaMemcpyHostToDevice,
                        s) != cudaSuccess ||
        cudaMemcpyAsync(ws + offsetof(WsHeader, stamp), m + plan->meta_bytes,
                        sizeof(unsigned long long), cudaMemcpyHostToDevice, s) != cudaSuccess)
        return OXD_ERR_CUDA;
    plan->bound_ws.store(workspace);
    return OXD_OK;
}

oxd_status oxd_prefill_plan_destroy(oxd_prefill_plan plan) {
    if (plan == nullptr) return OXD_ERR_INVALID_ARGUMENT;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (g_live.erase(plan) == 0) return OXD_ERR_PLAN_MISMATCH;
    }
    free_plan(plan);
    return OXD_OK;
}

oxd_status oxd_paged_prefill_run(oxd_prefill_plan plan, const void* q, const void* k_pages,
                                 const void* v_pages, const int32_t* qo_indptr,
                                 const int32_t* indptr, const int32_t* indices,
                                 const int32_t* last_page_len, float sm_scale, void* out,
                                 float* lse, void* workspace, size_t workspace_bytes,
                                 void* stream) {
    if (plan == nullptr || !alive(plan)) return OXD_ERR_PLAN_MISMATCH;
    if (q == nullptr || k_pages == nullptr || v_pages == nullptr || qo_indptr == nullptr ||
        indptr == nullptr || indices == nullptr || last_page_len == nullptr || out == nullptr ||
        workspace == nullptr)
        return OXD_ERR_INVALID_ARGUMENT;
    if (!std::isfinite(sm_scale)) return OXD_ERR_INVALID_ARGUMENT;
    const oxd_paged_prefill_desc& d = plan->desc;
    if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(out, 16) ||
        !aligned(qo_indptr, 4) || !aligned(indptr, 4) || !aligned(indices, 4) ||
        !aligned(last_page_len, 4) || !aligned(lse, 4) || !aligned(workspace, 256))
        return OXD_ERR_ALIGNMENT;
    if (workspace_bytes < plan->ws_bytes) return OXD_ERR_WORKSPACE_TOO_SMALL;
    const size_t rows = static_cast<size_t>(plan->nq) * d.num_qo_heads;
    const size_t pool =
        static_cast<size_t>(d.num_pages) * d.page_size * d.num_kv_heads * kHeadDim * 2;
    const size_t tab = (static_cast<size_t>(d.batch) + 1) * 4;
    const Span in[] = {span(q, rows * kHeadDim * 2),
                       span(k_pages, pool),
                       span(v_pages, pool),
                       span(qo_indptr, tab),
                       span(indptr, tab),
                       span(indices, static_cast<size_t>(plan->nnz) * 4),
                       span(last_page_len, static_cast<size_t>(d.batch) * 4)};
    const Span outs[] = {span(out, rows * kHeadDim * 2), lse ? span(lse, rows * 4) : Span{0, 0},
                         span(workspace, plan->ws_bytes)};
    for (const Span& o : outs)
        for (const Span& i : in)
            if (overlap(o, i)) return OXD_ERR_ALIAS;
    if (overlap(outs[0], outs[1]) || overlap(outs[0], outs[2]) || overlap(outs[1], outs[2]))
        return OXD_ERR_ALIAS;
    // operands are checked first (so every rejection above needs no GPU);
    // a host-only plan is never run
    if (plan->device < 0) return OXD_ERR_PLAN_MISMATCH;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) return OXD_ERR_CUDA;
    if (cur != plan->device) return OXD_ERR_PLAN_MISMATCH;

    CUtensorMap tk, tv, tq;
    if (!encode_kv_pool(&tk, k_pages, d.layout, d.page_size, d.num_kv_heads, d.num_pages) ||
        !encode_kv_pool(&tv, v_pages, d.layout, d.page_size, d.num_kv_heads, d.num_pages))
        return OXD_ERR_CUDA;
    if (plan->narrow) {
        // q as (d, head, token): a box is 64 columns x the G heads of one KV
        // head x the tile's query tokens
        const uint64_t dims[3] = {static_cast<uint64_t>(kHeadDim),
                                  static_cast<uint64_t>(d.num_qo_heads),
                                  static_cast<uint64_t>(plan->nq)};
        const uint64_t strides[2] = {static_cast<uint64_t>(kHeadDim) * 2,
                                     static_cast<uint64_t>(d.num_qo_heads) * kHeadDim * 2};
        const uint32_t box[3] = {64, static_cast<uint32_t>(plan->group),
                                 static_cast<uint32_t>(plan->tile_tokens)};
        if (!encode_bf16_map(&tq, q, 3, dims, strides, box)) return OXD_ERR_CUDA;
    }

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const bool bound = plan->bound_ws.load() == workspace;
    constexpr size_t kStampOff = offsetof(WsHeader, stamp);
    // an unbound run uploads the list with a zero stamp, which also ends any
    // binding of another plan to this workspace
    if (!bound && cudaMemcpyAsync(ws + kStampOff, static_cast<uint8_t*>(plan->meta) + kStampOff,
                                  plan->meta_bytes - kStampOff, cudaMemcpyHostToDevice,
                                  s) != cudaSuccess)
        return OXD_ERR_CUDA;

    PrefillParams p{};
    p.q = static_cast<const uint16_t*>(q);
    p.out = static_cast<uint16_t*>(out);
    p.lse = lse;
    p.qo_indptr = qo_indptr;
    p.indptr = indptr;
    p.indices = indices;
    p.last_page_len = last_page_len;
    p.units = reinterpret_cast<const PrefillUnit*>(ws + plan->off_units);
    p.ws_stamp = bound ? reinterpret_cast<const unsigned long long*>(ws + kStampOff) : nullptr;
    p.stamp = plan->stamp;
    p.clear_stamp = nullptr;  // the upload above already zeroed it
    p.part_o = reinterpret_cast<float*>(ws + plan->off_part_o);
    p.part_lse = reinterpret_cast<float*>(ws + plan->off_part_lse);
    p.n_states = plan->n_groups * plan->group;
    p.status = reinterpret_cast<unsigned long long*>(ws + offsetof(WsHeader, status));
    p.last_epoch = reinterpret_cast<uint32_t*>(ws + offsetof(WsHeader, last_epoch));
    p.epoch = next_run_epoch();
    p.n_units = plan->n_units;
    p.batch = d.batch;
    p.n_q_tokens = static_cast<int32_t>(plan->nq);
    p.nnz = plan->nnz;
    p.num_qo_heads = d.num_qo_heads;
    p.num_kv_heads = d.num_kv_heads;
    p.group = plan->group;
    p.tile_tokens = plan->tile_tokens;
    p.page_size = d.page_size;
    p.layout = d.layout;
    p.num_pages = d.num_pages;
    p.scale_log2 = sm_scale * 1.4426950408889634f;  // log2(e)
    p.wait_ns = d.wait_timeout_ns > 0 ? d.wait_timeout_ns : kWaitTimeoutNs;

    if (plan->ev_before != nullptr && cudaEventRecord(plan->ev_before, s) != cudaSuccess)
        return OXD_ERR_CUDA;
    if ((plan->narrow ? launch_prefill_narrow(tk, tv, tq, p, plan->n_units, s)
                      : launch_prefill(tk, tv, p, plan->n_units, s)) != cudaSuccess)
        return OXD_ERR_CUDA;
    if (plan->ev_after != nullptr && cudaEventRecord(plan->ev_after, s) != cudaSuccess)
        return OXD_ERR_CUDA;
    if (plan->n_entries > 0) {
        MergeParams mp{};
        mp.v = p.part_o;
        mp.s = p.part_lse;
        mp.out = p.out;
        mp.lse = lse;
        mp.entries = reinterpret_cast<const int4*>(ws + plan->off_entries);
        mp.ws_stamp = p.ws_stamp;
        mp.stamp = p.stamp;
        mp.n_rows = static_cast<int64_t>(rows);
        mp.n_states = p.n_states;
        mp.uniform = 0;
        mp.n = plan->n_entries;
        mp.S = 0;
        mp.R = plan->group;
        mp.D = kHeadDim;
        mp.s_to_ln = 0.693147180559945309f;  // partial LSEs are log2
        mp.max_count = plan->max_pieces;
        if (launch_split_merge(mp, nullptr, s, plan->ev_after == nullptr) != cudaSuccess)
            return OXD_ERR_CUDA;
    }
    return OXD_OK;
}

}  // extern "C"
