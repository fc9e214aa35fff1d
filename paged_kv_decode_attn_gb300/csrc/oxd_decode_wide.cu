// Paged-KV decode for large query groups (17..32 query heads per KV head,
// MQA-like) on the 5th-generation tensor cores of sm_103a.
//
// Operation: "FlashInfer parity matrix" page, "Admitted attention matrix",
// row "Paged batch decode" (MQA/GQA), with the F32 online softmax every
// attention row there fixes and the split partitions + F32 partial workspace
// of the "Single decode split-K" row. Same work list, stage records, checks,
// status words and partial-state format as paged_decode_kernel; only the
// arithmetic moves from mma.sync to tcgen05.
//
// One CTA serves all rows of a group (up to 32), three warps:
//   * producer (warp 2): TMA copies of each stage's K and V pages (64 tokens,
//     two 64-column halves of 128-byte swizzled rows each) into a ring of
//     three stages, and of the group's query rows into a query tile on a
//     unit's first stage;
//   * MMA warp (warp 1, one thread): S = Q K^T into one of two TMEM score
//     buffers (M = 128 rows, the group's rows first, N = 64 tokens, K = 128),
//     then, once the softmax has written P, O += P V with P read from TMEM
//     as the A operand and V as an MN-major B operand (N = 128 dims, K = 64
//     tokens); each MMA is issued as soon as its inputs are ready, so the
//     score MMA of the next stage runs while the softmax works;
//   * softmax warp (warp 0): lane r owns query row r (TMEM lane r): it reads
//     the stage's 64 scores, updates the running maximum and denominator,
//     writes P as bf16 over its scores, rescales O in TMEM only when the
//     maximum grew by more than 2^8 (otherwise the stale maximum is kept,
//     so P stays below 256), and at a unit's end writes out/lse or the F32
//     partial state.
// The query tile holds only the group's 32 rows; the score MMA's rows 32..127
// read whatever follows in shared memory and their results are never read.
// V rows of tokens past the end of a unit are zeroed before its last PV, so
// stale or NaN pool slots never reach O.
// Every mbarrier wait gives up after about a second (OXD_DEVICE_WAIT_TIMEOUT);
// before the CTA returns, the MMAs and copies already issued are drained and
// the tensor memory is released.
#include <cuda_bf16.h>

#include <atomic>
#include <type_traits>

#include "oxd_internal.h"
#include "oxd_ptx.cuh"
#include "oxd_tcgen05.cuh"

namespace oxd {
namespace {

constexpr int kWRows = 32;                       // query rows a CTA serves
constexpr int kWStageTokens = 64;
constexpr int kWStages = 3;
constexpr int kWThreads = 96;
constexpr int kWHalf = kWStageTokens * 128;      // one 64-column half of K or V: 8 KB
constexpr int kWStageBytes = 4 * kWHalf;         // K halves, then V halves: 32 KB
constexpr int kWQHalf = kWRows * 128;            // 4 KB
constexpr int kWQOff = 0;                        // query tile: two halves
constexpr int kWRingOff = 2 * kWQHalf;           // 8 KB
constexpr int kWCtlOff = kWRingOff + kWStages * kWStageBytes;
constexpr uint32_t kWTmemCols = 256;             // O [0,128), S0 [128,192), S1 [192,256)
static_assert(kWRingOff % 1024 == 0 && kWStageBytes % 1024 == 0, "swizzle atoms aligned");
// The score MMA reads 128 rows (16 KB) from each query half: both spans must
// lie inside the CTA's shared memory.
static_assert(kWQOff + kWQHalf + 16 * 1024 <= kWCtlOff, "query-tile MMA rows in bounds");

struct WStageRec {
    int b, hkv, valid, n_stages, s, slot, row0, nrows;
};

struct WCtl {
    WStageRec rec[kWStages];
    uint64_t full[kWStages];
    uint64_t empty[kWStages];
    uint64_t s_ready[2];
    uint64_t p_ready[2];
    uint64_t o_ready[4];  // PV(k) completes phase k / 4 of o_ready[k % 4]
    uint64_t q_free;
    uint64_t mma_done;
    int issued[kWStages];
    uint32_t tmem;
    int flags[4];  // [0] abort
};
constexpr int kWSmemBytes = 1024 /* alignment slack */ + kWCtlOff + static_cast<int>(sizeof(WCtl));

// ------------------------------------------------------------------ the kernel

template <class WL>
__global__ void __launch_bounds__(kWThreads)
    paged_decode_wide_kernel(const __grid_constant__ CUtensorMap tmap_k,
                             const __grid_constant__ CUtensorMap tmap_v,
                             const __grid_constant__ CUtensorMap tmap_q,
                             const __grid_constant__ DecodeParams p,
                             const __grid_constant__ WL work) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    WCtl& ctl = *reinterpret_cast<WCtl*>(sm + kWCtlOff);
    volatile int* flags = ctl.flags;
    const uint32_t s_base = smem_addr(sm);
    const uint32_t s_q = s_base + kWQOff;
    auto ring_k = [&](int slot) { return s_base + kWRingOff + slot * kWStageBytes; };
    auto ring_v = [&](int slot) { return s_base + kWRingOff + slot * kWStageBytes + 2 * kWHalf; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ps = p.page_size;
    const int pages_per_stage = kWStageTokens / ps;
    const int G = p.group;
    const int4* units = p.units;
    const int32_t* cta_begin = nullptr;
    if constexpr (std::is_same<WL, WorkList>::value) {
        if (units == nullptr) {
            units = work.unit;
            cta_begin = work.cta_begin;
        }
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < kWStages; ++s) {
            mbar_init(&ctl.full[s], 1);
            mbar_init(&ctl.empty[s], 1);
            ctl.issued[s] = 0;
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctl.s_ready[i], 1);
            mbar_init(&ctl.p_ready[i], 1);
        }
        for (int i = 0; i < 4; ++i) mbar_init(&ctl.o_ready[i], 1);
        mbar_init(&ctl.q_free, 1);
        mbar_init(&ctl.mma_done, 1);
        flags[0] = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile(
            "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                smem_addr(&ctl.tmem)),
            "r"(kWTmemCols)
            : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (warp == 2 && lane == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
        prefetch_tmap(&tmap_q);
    }
    // A programmatic dependent of the kernel before it (pdl = 1) touches no
    // global memory before this wait; launched plainly it returns at once.
    grid_dependency_wait();
    if (threadIdx.x == 0) {
        if (blockIdx.x == 0) {
            *p.last_epoch = p.epoch;  // whose status the word may hold
            // an unbound run ends any binding of the workspace it writes
            if (p.clear_stamp != nullptr) *p.clear_stamp = 0ull;
        }
        // The merge kernel, when the plan has one, may be scheduled now; it
        // waits for this grid to complete before it reads anything.
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem;
    const uint32_t t_o = tmem;
    auto t_s = [&](int buf) { return tmem + 128u + 64u * static_cast<uint32_t>(buf); };

    if (warp == 2) {
        // ================================================ producer warp
        struct Unit {
            int unit;
            int4 it;
            int win, nxt;  // page indices [0, 32) and [32, 64) of the unit, by lane
        };
        // A bound workspace is used only while it still carries this plan's
        // stamp; every unit is bounds-checked before it is used.
        int u_begin, u_end;
        int4 first_it = make_int4(0, 0, 0, 0);
        const bool rec_first = cta_begin == nullptr;
        if (rec_first) {
            const int4 r0 = __ldg(p.cta_rec + 2 * blockIdx.x);
            first_it = __ldg(p.cta_rec + 2 * blockIdx.x + 1);
            u_begin = r0.x;
            u_end = r0.y;
        } else {
            u_begin = cta_begin[blockIdx.x];
            u_end = cta_begin[blockIdx.x + 1];
        }
        if (p.ws_stamp != nullptr) {
            int ok_stamp = 1;
            if (lane == 0) ok_stamp = *p.ws_stamp == p.stamp ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, ok_stamp, 0)) {
                if (lane == 0) record_status(p.status, p.epoch, kDevicePlanMismatch);
                u_begin = u_end = 0;
            }
        }
        if (u_begin < 0 || u_end > p.n_units || u_begin > u_end) {
            if (lane == 0) record_status(p.status, p.epoch, kDevicePlanMismatch);
            u_begin = u_end = 0;
        }
        auto pages_of = [](const int4& it) { return it.y & ((1 << kUnitPagesBits) - 1); };
        auto load_item = [&](Unit& u) {
            if (u.unit < u_end) u.it = units[u.unit];
        };
        auto load_idx = [&](Unit& u) {
            u.win = u.nxt = 0;
            if (u.unit < u_end && u.it.x >= 0 &&
                static_cast<int64_t>(u.it.x) + pages_of(u.it) <= p.nnz) {
                const int32_t* idx = p.indices + u.it.x;
                const int n = pages_of(u.it);
                if (lane < n) u.win = __ldg(idx + lane);
                if (32 + lane < n) u.nxt = __ldg(idx + 32 + lane);
            }
        };
        int g = 0;        // ring position
        int started = 0;  // units whose stages were issued
        bool ok = true;
        Unit cur;
        cur.unit = u_begin;
        if (rec_first)
            cur.it = first_it;
        else
            load_item(cur);
        load_idx(cur);
        while (cur.unit < u_end) {
            Unit nx;
            nx.unit = cur.unit + 1;
            bool nx_item = false, nx_idx = false;
            const int4 it = cur.it;
            const int n_pages = pages_of(it);
            const int last_len = (it.y >> kUnitPagesBits) & 0x7f;  // 0: not the last page
            const bool first_page = it.y < 0;                         // bit 31
            const int b = it.z & ((1 << kUnitBBits) - 1);
            const bool half_bit = ((it.z >> kUnitBBits) & 1) != 0;   // never set for this kernel
            const int hkv = static_cast<int>(static_cast<uint32_t>(it.z) >> (kUnitBBits + 1));
            const int valid = last_len ? (n_pages - 1) * ps + last_len : n_pages * ps;
            int n_stages = (n_pages + pages_per_stage - 1) / pages_per_stage;
            const bool unit_ok = n_pages >= 1 && it.x >= 0 &&
                                 static_cast<int64_t>(it.x) + n_pages <= p.nnz && b < p.batch &&
                                 hkv < p.num_kv_heads && !half_bit && it.w >= -1 &&
                                 it.w < p.n_slots && last_len <= ps;
            if (!unit_ok) {
                // not a unit of this plan: skip it (its outputs stay unwritten)
                if (lane == 0) record_status(p.status, p.epoch, kDevicePlanMismatch);
                n_stages = 0;
            }
            int ip0 = 0, ip1 = 0, lst = 0;
            if (lane == 0 && unit_ok) {
                if (first_page) ip0 = p.indptr[b];
                if (last_len) {
                    ip1 = p.indptr[b + 1];
                    lst = p.last_page_len[b];
                }
            }
            // An index outside [0, num_pages) is recorded and replaced by page
            // 0, so every copy stays inside the pool.
            const int32_t* idx = p.indices + it.x;
            int win = cur.win, nxt = cur.nxt;
            int win_base = 0;
            bool bad = win < 0 || static_cast<int64_t>(win) >= p.num_pages;
            if (__any_sync(0xffffffffu, bad) && lane == 0)
                record_status(p.status, p.epoch, kDeviceBadPage);
            win = bad ? 0 : win;
            for (int s = 0; s < n_stages; ++s, ++g) {
                const int slot = g % kWStages;
                const int pg0 = s * pages_per_stage;
                const int npg = min(pages_per_stage, n_pages - pg0);
                if (pg0 >= win_base + 32) {
                    win = nxt;
                    win_base += 32;
                    nxt = win_base + 32 + lane < n_pages ? __ldg(idx + win_base + 32 + lane) : 0;
                    bad = win < 0 || static_cast<int64_t>(win) >= p.num_pages;
                    if (__any_sync(0xffffffffu, bad) && lane == 0)
                        record_status(p.status, p.epoch, kDeviceBadPage);
                    win = bad ? 0 : win;
                }
                int okw = 1;
                if (lane == 0) {
                    if (g >= kWStages)
                        okw = mbar_wait_tc(&ctl.empty[slot], ((g / kWStages) + 1) & 1, flags, p.wait_ns)
                                  ? 1
                                  : 0;
                    // the query tile is rewritten only after the previous
                    // unit's last score MMA has read it
                    if (okw && s == 0 && started > 0)
                        okw = mbar_wait_tc(&ctl.q_free, (started - 1) & 1, flags, p.wait_ns) ? 1 : 0;
                }
                if (!__shfl_sync(0xffffffffu, okw, 0)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    WStageRec* r = &ctl.rec[slot];
                    r->b = b;
                    r->hkv = hkv;
                    r->valid = valid;
                    r->n_stages = n_stages;
                    r->s = s;
                    r->slot = it.w;
                    r->row0 = 0;
                    r->nrows = G;
                    const uint32_t qbytes = s == 0 ? 2u * kWQHalf : 0u;
                    mbar_arrive_expect_tx(&ctl.full[slot],
                                          npg * ps * kHeadDim * 2 * 2 + qbytes);
                    if (s == 0) {
                        const int qrow = b * p.num_qo_heads + hkv * G;
                        tma_load_2d(s_q, &tmap_q, &ctl.full[slot], 0, qrow);
                        tma_load_2d(s_q + kWQHalf, &tmap_q, &ctl.full[slot], 64, qrow);
                    }
                }
                const uint32_t tk = ring_k(slot);
                const uint32_t tv = ring_v(slot);
                const int ca = p.layout == 0 ? hkv : 0;  // coordinates (d, A, B, page):
                const int cb = p.layout == 0 ? 0 : hkv;  // NHD (d, head, token, page)
                {                                        // HND (d, token, head, page)
                    // One copy per (page, tensor, 64-column half), one lane each:
                    // lane 4j + 2t + h copies half h of tensor t (K, V) of page j.
                    const int j = lane >> 2;
                    const int page = __shfl_sync(0xffffffffu, win, (pg0 - win_base + j) & 31);
                    if (lane < 4 * npg) {
                        const uint32_t off = j * ps * 128 + ((lane & 1) ? kWHalf : 0);
                        tma_load_4d(((lane & 2) ? tv : tk) + off, (lane & 2) ? &tmap_v : &tmap_k,
                                    &ctl.full[slot], (lane & 1) * 64, ca, cb, page);
                    }
                }
                if (lane == 0) ctl.issued[slot] += 1;
                if (s == 0) {
                    load_item(nx);
                    nx_item = true;
                } else if (s == 1) {
                    load_idx(nx);
                    nx_idx = true;
                }
            }
            if (!ok) break;
            if (n_stages > 0) ++started;
            if (!nx_item) load_item(nx);
            if (!nx_idx) load_idx(nx);
            if (lane == 0 && unit_ok &&
                ((first_page && ip0 != it.x) ||
                 (last_len && (ip1 != it.x + n_pages || lst != last_len))))
                record_status(p.status, p.epoch, kDevicePlanMismatch);
            cur = nx;
        }
        if (ok) {
            // End marker: a stage whose record says s = -1, completed by a
            // plain arrive (no bytes).
            const int slot = g % kWStages;
            int okw = 1;
            if (lane == 0) {
                if (g >= kWStages)
                    okw = mbar_wait_tc(&ctl.empty[slot], ((g / kWStages) + 1) & 1, flags, p.wait_ns)
                                  ? 1
                                  : 0;
                if (okw) {
                    ctl.rec[slot].s = -1;
                    mbar_arrive(&ctl.full[slot]);
                    ctl.issued[slot] += 1;
                }
            }
            ok = __shfl_sync(0xffffffffu, okw, 0) != 0;
        }
        if (!ok && lane == 0) {
            flags[0] = 1;
            record_status(p.status, p.epoch, kDeviceWaitTimeout);
        }
    } else if (warp == 1) {
        // ================================================ MMA warp
        if (lane == 0) {
            constexpr uint32_t kIdQK = umma_idesc(128, kWStageTokens, 0);
            constexpr uint32_t kIdPV = umma_idesc(128, kHeadDim, 1);
            // Two kinds of work, issued as soon as each is ready: the score
            // MMA of stage gq (once its K/V have landed and its score buffer
            // is free, i.e. the PV of stage gq - 2 was issued) and the PV of
            // stage gp (once the softmax has written its P).
            int gq = 0, gp = 0;
            int slot_even = 0, slot_odd = 0;    // ring slot of the pending stages,
            bool first_even = false, first_odd = false;  // by stage parity
            bool ended = false, ok = true, issued_any = false;
            uint64_t idle_since = global_ns();
            while (!(ended && gp == gq)) {
                bool progress = false;
                if (!ended && gq < gp + 2 &&
                    mbar_try_wait(&ctl.full[gq % kWStages], (gq / kWStages) & 1)) {
                    const int slot = gq % kWStages;
                    const WStageRec rec = ctl.rec[slot];
                    if (rec.s < 0) {
                        ended = true;
                    } else {
                        tc_fence_after();
                        // S = Q K^T: K = 128 in steps of 16 (32 bytes of a
                        // 128-byte swizzled row; columns 64..127 in the other
                        // half)
                        const uint32_t k0 = ring_k(slot);
                        for (int ks = 0; ks < kHeadDim / 16; ++ks) {
                            const uint32_t h = static_cast<uint32_t>(ks >> 2), kk = ks & 3;
                            const uint64_t ad = umma_sdesc(s_q + h * kWQHalf + kk * 32, 16, 1024);
                            const uint64_t bd = umma_sdesc(k0 + h * kWHalf + kk * 32, 16, 1024);
                            umma_ss(t_s(gq & 1), ad, bd, kIdQK, ks > 0 ? 1u : 0u);
                        }
                        issued_any = true;
                        umma_commit(&ctl.s_ready[gq & 1]);
                        if (rec.s == rec.n_stages - 1) umma_commit(&ctl.q_free);
                        if (gq & 1) {
                            slot_odd = slot;
                            first_odd = rec.s == 0;
                        } else {
                            slot_even = slot;
                            first_even = rec.s == 0;
                        }
                        ++gq;
                    }
                    progress = true;
                }
                if (gp < gq && mbar_try_wait(&ctl.p_ready[gp & 1], (gp >> 1) & 1)) {
                    tc_fence_after();
                    // O += P V: 16 tokens a step = two 8-row groups (1024 B
                    // apart); the two 64-column halves of V are kWHalf apart
                    const int slot = (gp & 1) ? slot_odd : slot_even;
                    const bool first = (gp & 1) ? first_odd : first_even;
                    const uint32_t v0 = ring_v(slot);
                    for (int ks = 0; ks < kWStageTokens / 16; ++ks) {
                        const uint64_t bd = umma_sdesc(v0 + ks * 2048, kWHalf, 1024);
                        umma_ts(t_o, t_s(gp & 1) + 8u * ks, bd, kIdPV,
                                (ks > 0 || !first) ? 1u : 0u);
                    }
                    umma_commit(&ctl.empty[slot]);  // K and V of the slot are consumed
                    umma_commit(&ctl.o_ready[gp & 3]);
                    ++gp;
                    progress = true;
                }
                if (progress) {
                    idle_since = global_ns();
                } else {
                    __nanosleep(32);  // leave the issue slots to the other warps
                    if (flags[0] ||
                        global_ns() - idle_since > static_cast<uint64_t>(p.wait_ns)) {
                        ok = false;
                        break;
                    }
                }
            }
            if (!ok) {
                flags[0] = 1;
                record_status(p.status, p.epoch, kDeviceWaitTimeout);
            }
            if (issued_any) {
                // every MMA completes before the tensor memory is released
                umma_commit(&ctl.mma_done);
                mbar_wait_tc(&ctl.mma_done, 0, nullptr, kWaitTimeoutNs);
            }
        }
        __syncwarp();
    } else {
        // ================================================ softmax warp
        // Lane r owns query row r, which is TMEM lane r. Every lane waits on
        // each barrier itself; the results are AND-ed over the warp so the
        // lanes always take the same path through the collective TMEM
        // instructions.
        auto wait_all = [&](uint64_t* bar, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait_tc(bar, parity, flags, p.wait_ns));
        };
        const float sc = p.scale_log2;
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int g = 0;; ++g) {
            const int slot = g % kWStages;
            if (!wait_all(&ctl.full[slot], (g / kWStages) & 1)) {
                ok = false;
                break;
            }
            const WStageRec rec = ctl.rec[slot];
            if (rec.s < 0) break;
            if (!wait_all(&ctl.s_ready[g & 1], (g >> 1) & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[64];
            tmem_ld64(t_s(g & 1), sr);
            const int nvalid = min(kWStageTokens, rec.valid - rec.s * kWStageTokens);
            // A full stage (the common case) takes the maximum over the raw
            // scores and folds the scale into the exponent's FMA; a stage
            // past the unit's end is scaled and masked first.
            const bool whole = nvalid == kWStageTokens && sc > 0.f;
            float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (whole) {
#pragma unroll
                for (int j = 0; j < 64; j += 2)
                    mq[(j >> 1) & 3] = max3(mq[(j >> 1) & 3], __uint_as_float(sr[j]),
                                            __uint_as_float(sr[j + 1]));
            } else {
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    const float x = j < nvalid ? __uint_as_float(sr[j]) * sc : -INFINITY;
                    sr[j] = __float_as_uint(x);
                    mq[j & 3] = fmaxf(mq[j & 3], x);
                }
            }
            float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
            if (whole) mx *= sc;
            const bool first = rec.s == 0;
            float alpha = 1.f;
            bool rescale = false;
            if (first) {
                m_ref = mx;
                l = 0.f;
            } else if (mx > m_ref + 8.f && lane < rec.nrows) {
                alpha = fast_exp2(m_ref - mx);
                m_ref = mx;
                l *= alpha;
                rescale = true;
            }
            uint32_t pk[32];
            float lq[4] = {0.f, 0.f, 0.f, 0.f};
            if (whole) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    float x0, x1;
                    fma2(__uint_as_float(sr[2 * j]), __uint_as_float(sr[2 * j + 1]), sc, -m_ref,
                         x0, x1);
                    const float p0 = fast_exp2(x0);
                    const float p1 = fast_exp2(x1);
                    add2(lq[(j & 1) * 2], lq[(j & 1) * 2 + 1], p0, p1);
                    pk[j] = pack_bf16x2(p0, p1);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float p0 = fast_exp2(__uint_as_float(sr[2 * j]) - m_ref);
                    const float p1 = fast_exp2(__uint_as_float(sr[2 * j + 1]) - m_ref);
                    lq[j & 3] += p0 + p1;
                    pk[j] = pack_bf16x2(p0, p1);
                }
            }
            l += (lq[0] + lq[1]) + (lq[2] + lq[3]);
            tmem_st32(t_s(g & 1), pk);
            tmem_wait_st();
            // P(g) is published without waiting for PV(g - 1): MMAs from one
            // thread run in issue order, so PV(g) follows it anyway. Only an
            // O rescale waits for PV(g - 1). Parity waits on the four
            // o_ready barriers are exact: s_ready(g) means every MMA issued
            // before QK(g), PV(g - 2) included, has completed, so PV(g - 5)
            // is done, and PV(g + 3) needs P(g + 3), not yet written.
            if (__any_sync(0xffffffffu, rescale)) {
                if (!wait_all(&ctl.o_ready[(g - 1) & 3], ((g - 1) >> 2) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int c0 = 0; c0 < kHeadDim; c0 += 64) {
                    uint32_t o[64];
                    tmem_ld64(t_o + c0, o);
                    uint32_t w0[32], w1[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        w0[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                        w1[j] = __float_as_uint(__uint_as_float(o[32 + j]) * alpha);
                    }
                    tmem_st32(t_o + c0, w0);
                    tmem_st32(t_o + c0 + 32, w1);
                }
                tmem_wait_st();
            }
            const bool last = rec.s == rec.n_stages - 1;
            if (last && nvalid < kWStageTokens) {
                // zero V rows past the unit's end (whole 128-byte rows, so the
                // swizzle does not matter)
                uint8_t* v0 = sm + kWRingOff + slot * kWStageBytes + 2 * kWHalf;
                const int n16 = (kWStageTokens - nvalid) * 16;
                for (int i = lane; i < n16; i += 32) {
                    const int row = nvalid + (i >> 4), c = i & 15;
                    *reinterpret_cast<uint4*>(v0 + (c >> 3) * kWHalf + row * 128 + (c & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.p_ready[g & 1]);
            if (last) {
                // ---- unit epilogue: O / l, once PV(g) is done
                if (!wait_all(&ctl.o_ready[g & 3], (g >> 2) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float inv = 1.f / l;
                const float lse2 = m_ref + __log2f(l);
                const bool row_ok = lane < rec.nrows;
                const int hq = rec.hkv * G + lane;
                for (int c0 = 0; c0 < kHeadDim; c0 += 64) {
                    uint32_t o[64];
                    tmem_ld64(t_o + c0, o);
                    if (!row_ok) continue;
                    if (rec.slot < 0) {
                        uint16_t* dst = p.out +
                                        (static_cast<size_t>(rec.b) * p.num_qo_heads + hq) *
                                            kHeadDim + c0;
#pragma unroll
                        for (int j = 0; j < 64; j += 8) {
                            uint4 w;
                            w.x = pack_bf16x2(__uint_as_float(o[j]) * inv,
                                              __uint_as_float(o[j + 1]) * inv);
                            w.y = pack_bf16x2(__uint_as_float(o[j + 2]) * inv,
                                              __uint_as_float(o[j + 3]) * inv);
                            w.z = pack_bf16x2(__uint_as_float(o[j + 4]) * inv,
                                              __uint_as_float(o[j + 5]) * inv);
                            w.w = pack_bf16x2(__uint_as_float(o[j + 6]) * inv,
                                              __uint_as_float(o[j + 7]) * inv);
                            *reinterpret_cast<uint4*>(dst + j) = w;
                        }
                    } else {
                        // partial states are [slot][G][128]
                        float* dst = p.part_o +
                                     (static_cast<size_t>(rec.slot) * G + lane) * kHeadDim + c0;
#pragma unroll
                        for (int j = 0; j < 64; j += 4)
                            *reinterpret_cast<float4*>(dst + j) =
                                make_float4(__uint_as_float(o[j]) * inv,
                                            __uint_as_float(o[j + 1]) * inv,
                                            __uint_as_float(o[j + 2]) * inv,
                                            __uint_as_float(o[j + 3]) * inv);
                    }
                }
                if (row_ok) {
                    if (rec.slot < 0) {
                        if (p.lse != nullptr)
                            p.lse[static_cast<size_t>(rec.b) * p.num_qo_heads + hq] = lse2 * kLn2;
                    } else {
                        p.part_lse[static_cast<size_t>(rec.slot) * G + lane] = lse2;
                    }
                }
            }
        }
        if (!ok && lane == 0) {
            flags[0] = 1;
            record_status(p.status, p.epoch, kDeviceWaitTimeout);
        }
    }
    tc_fence_before();
    __syncthreads();  // every warp has left its loop; the MMAs have completed

    if (flags[0] && threadIdx.x == 0) {
        // Aborted: wait (bounded) for the copies already issued, then leave.
        for (int s = 0; s < kWStages; ++s)
            if (ctl.issued[s] > 0)
                mbar_wait_tc(&ctl.full[s], (ctl.issued[s] - 1) & 1, nullptr, kWaitTimeoutNs);
    }
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kWTmemCols)
                     : "memory");
    }
}

template <class WL>
cudaError_t ensure_wide_attribute() {
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit != 0 && (done.load(std::memory_order_relaxed) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(paged_decode_wide_kernel<WL>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kWSmemBytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_relaxed);
    return e;
}

}  // namespace

VariantShape wide_shape() { return {kWThreads, kWStageTokens, kWStages, kWSmemBytes}; }

// Resident CTAs per SM from shared memory, threads and tensor-memory columns.
// The occupancy query answers 1 for any kernel that uses tcgen05; two of
// these CTAs (256 TMEM columns each) do run side by side on one SM.
cudaError_t wide_occupancy(int* n) {
    cudaError_t e = ensure_wide_attribute<WorkList>();
    if (e != cudaSuccess) return e;
    int dev = 0, smem_sm = 0, reserved = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
        cudaSuccess)
        return e;
    if ((e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) !=
        cudaSuccess)
        return e;
    const int by_smem = smem_sm / (kWSmemBytes + reserved);
    const int by_tmem = 512 / static_cast<int>(kWTmemCols);
    const int by_threads = 2048 / kWThreads;
    *n = max(1, min(by_smem, min(by_tmem, by_threads)));
    return cudaSuccess;
}

cudaError_t launch_decode_wide(const CUtensorMap& tk, const CUtensorMap& tv,
                               const CUtensorMap& tq, const DecodeParams& p, const WorkList* w,
                               int grid, cudaStream_t stream, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kWThreads);
    cfg.dynamicSmemBytes = kWSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    // pdl: a programmatic dependent of the kernel before it on the stream
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (w != nullptr) {
        cudaError_t e = ensure_wide_attribute<WorkList>();
        if (e != cudaSuccess) return e;
        return cudaLaunchKernelEx(&cfg, paged_decode_wide_kernel<WorkList>, tk, tv, tq, p, *w);
    }
    cudaError_t e = ensure_wide_attribute<NoList>();
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, paged_decode_wide_kernel<NoList>, tk, tv, tq, p, NoList{0});
}

}  // namespace oxd
