// Narrow paged causal prefill for sm_103a: 128-row tiles, two CTAs a SM.
//
// Operation: "FlashInfer parity matrix" page, "Admitted attention matrix",
// row "Paged causal prefill" (BF16, D128, causal, NHD/HND pages through the
// same block tables as decode, split pieces with a caller-owned F32
// workspace). It serves the prefills whose 256-row plan would leave SMs
// idle (short ones, such as the pages' own shape: smaller tiles, two CTAs a
// SM and 64-token stages start and finish sooner), and the cascade decode's
// shared-prefix tiles ("Cascade inference" page): a sharing group's
// requests, one query token each, attend the group's common prefix with no
// mask, their partial states going to the decode's merge. Those start in
// the decode kernel's tail as each decode CTA retires: this kernel's
// footprint (112 KB of shared memory, 256 tensor-memory columns) lets one
// start beside a decode CTA still running, where the two-half 256-row
// kernel needs a whole SM.
//
// A tile is up to T = 128 / G consecutive query tokens of one request with
// the G query heads of one KV head each: 128 MMA rows, row r = token r / G,
// head r % G. One CTA runs one piece of a tile's cached-token range (a whole
// range, or one of the pieces of a split tile); six warps:
//   * producer (warp 5): on the first stage the tile's query rows through a
//     3-D tensor map (d, head, token) with a box of 64 x G x T; per stage of
//     64 cached tokens one TMA copy per (page, tensor, 64-column half) into a
//     ring of stages, laid out [half][64 tokens][128 B] with the 128-byte
//     swizzle;
//   * MMA warp (warp 4, one thread): S = Q K^T into one of two TMEM score
//     buffers (M = 128, N = 64, K = 128), then O += P V with P read from
//     TMEM (N = 128, K = 64), each issued as soon as its inputs are ready;
//   * softmax warps (warps 0-3): thread r of the warpgroup owns row r (TMEM
//     lane r). Per stage it loads the row's 64 scores, masks the tokens past
//     its position (and past the piece), keeps a running maximum that is
//     raised only when a score exceeds it by more than 2^8 (then O is
//     rescaled in TMEM, after the previous PV), writes P as bf16 over its
//     scores and publishes it without waiting for the previous PV (the MMAs
//     run in issue order), and at the end writes out/lse, or the F32 partial
//     state of the piece.
// V rows past the piece's last cached token are zeroed before its last PV.
// Every wait is bounded (OXD_DEVICE_WAIT_TIMEOUT); on abort the MMAs and
// copies in flight are drained before the tensor memory is released.
#include <cuda_bf16.h>

#include <atomic>

#include "oxd_internal.h"
#include "oxd_prefill.h"
#include "oxd_ptx.cuh"
#include "oxd_tcgen05.cuh"

namespace oxd {
namespace {

constexpr int kPKStages = 3;     // K ring: a slot is free once its score MMA is done
constexpr int kPVStages = 2;     // V ring: a slot is free once its PV is done
constexpr int kPThreads = 224;   // 4 softmax warps, MMA warp, K producer, V producer
constexpr int kPSoftmaxThreads = 128;
constexpr int kPHalf = kNarrowStageTokens * 128;  // one 64-column half of K or V: 8 KB
constexpr int kPSlotBytes = 2 * kPHalf;            // K or V of one stage: 16 KB
constexpr int kPQHalf = kNarrowRows * 128;        // 16 KB
constexpr int kPQOff = 0;
constexpr int kPKOff = 2 * kPQHalf;
constexpr int kPVOff = kPKOff + kPKStages * kPSlotBytes;
constexpr int kPCtlOff = kPVOff + kPVStages * kPSlotBytes;  // 112 KB of operands
constexpr uint32_t kPTmemCols = 256;  // O [0,128), S0 [128,192), S1 [192,256)
static_assert(kPKOff % 1024 == 0 && kPVOff % 1024 == 0 && kPSlotBytes % 1024 == 0,
              "swizzle atoms aligned");

struct PCtl {
    uint64_t kfull[kPKStages];
    uint64_t kempty[kPKStages];
    uint64_t vfull[kPVStages];
    uint64_t vempty[kPVStages];
    uint64_t s_ready[2];
    uint64_t p_ready[2];
    uint64_t o_ready[4];  // PV(g) completes phase g / 4 of o_ready[g % 4]
    uint64_t mma_done;
    int kissued[kPKStages];
    int vissued[kPVStages];
    uint32_t tmem;
    int flags[4];  // [0] abort, [1] the unit is usable
};
// The dynamic shared memory starts 1024-byte aligned (checked in the kernel),
// so no alignment slack: two CTAs fit one SM.
constexpr int kPSmemBytes = kPCtlOff + static_cast<int>(sizeof(PCtl));

__global__ void __launch_bounds__(kPThreads)
    paged_prefill_narrow_kernel(const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v,
                         const __grid_constant__ CUtensorMap tmap_q,
                         const __grid_constant__ PrefillParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw;
    PCtl& ctl = *reinterpret_cast<PCtl*>(sm + kPCtlOff);
    volatile int* flags = ctl.flags;
    const uint32_t s_base = smem_addr(sm);
    const uint32_t s_q = s_base + kPQOff;
    auto ring_k = [&](int slot) { return s_base + kPKOff + slot * kPSlotBytes; };
    auto ring_v = [&](int slot) { return s_base + kPVOff + slot * kPSlotBytes; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ps = p.page_size;
    const int G = p.group;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPKStages; ++s) {
            mbar_init(&ctl.kfull[s], 1);
            mbar_init(&ctl.kempty[s], 1);
            ctl.kissued[s] = 0;
        }
        for (int s = 0; s < kPVStages; ++s) {
            mbar_init(&ctl.vfull[s], 1);
            mbar_init(&ctl.vempty[s], 1);
            ctl.vissued[s] = 0;
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctl.s_ready[i], 1);
            mbar_init(&ctl.p_ready[i], 4);  // one arrival per softmax warp
        }
        for (int i = 0; i < 4; ++i) mbar_init(&ctl.o_ready[i], 1);
        mbar_init(&ctl.mma_done, 1);
        flags[0] = 0;
        fence_mbar_init();
        if (blockIdx.x == 0) {
            *p.last_epoch = p.epoch;
            if (p.clear_stamp != nullptr) *p.clear_stamp = 0ull;
        }
        // the unit, checked before anything uses it (and the operand
        // buffers' alignment, which the swizzled copies need)
        int ok = (p.ws_stamp == nullptr || *p.ws_stamp == p.stamp) && (s_base & 1023u) == 0;
        if (ok && static_cast<int>(blockIdx.x) < p.n_units) {
            const PrefillUnit u = p.units[blockIdx.x];
            const int T = p.tile_tokens;
            ok = u.n_pages >= 1 && u.idx_begin >= 0 &&
                 static_cast<int64_t>(u.idx_begin) + u.n_pages <= p.nnz && u.kv_valid >= 1 &&
                 u.kv_begin >= 0 && (u.kv_begin % kNarrowStageTokens) == 0 &&
                 static_cast<int64_t>(u.kv_begin % ps + u.kv_valid) <=
                     static_cast<int64_t>(u.n_pages) * ps &&
                 u.b >= 0 && u.b < p.batch && u.hkv >= 0 && u.hkv < p.num_kv_heads &&
                 u.n_tok >= 1 && u.n_tok <= T && u.q_begin >= 0 &&
                 u.q_begin + u.n_tok <= p.n_q_tokens && u.p0 >= 0 && u.n_pieces >= 1 &&
                 u.piece >= 0 && u.piece < u.n_pieces;
            if (ok && u.n_pieces > 1)
                ok = u.state >= 0 &&
                     (static_cast<int64_t>(u.state) +
                      static_cast<int64_t>(u.n_tok - 1) * u.n_pieces + u.piece + 1) *
                             G <=
                         p.n_states;
        } else {
            ok = 0;
        }
        if (!ok) record_status(p.status, p.epoch, kDevicePlanMismatch);
        flags[1] = ok;
    }
    if (warp == 4) {
        asm volatile(
            "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                smem_addr(&ctl.tmem)),
            "r"(kPTmemCols)
            : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (warp == 5 && lane == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
        prefetch_tmap(&tmap_q);
    }
    // The merge kernel, when the plan has one, may be scheduled now; it waits
    // for this grid to complete before it reads anything.
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem;
    const uint32_t t_o = tmem;
    auto t_s = [&](int buf) { return tmem + 128u + 64u * static_cast<uint32_t>(buf); };
    const bool usable = flags[1] != 0;
    PrefillUnit u{};
    if (usable) u = p.units[blockIdx.x];
    const int n_st = usable ? (u.kv_valid + kNarrowStageTokens - 1) / kNarrowStageTokens : 0;

    if (warp >= 5) {
        // ================================================ producer warps
        // warp 5: the query tile and K; warp 6: V. Lane 2j + h copies half h
        // of page j of the stage.
        const bool is_k = warp == 5;
        const int pps = kNarrowStageTokens / ps;  // pages per stage (divides 32)
        const int32_t* idx = p.indices + u.idx_begin;
        int win = 0, nxt = 0, win_base = 0;
        if (n_st > 0) {
            if (lane < u.n_pages) win = __ldg(idx + lane);
            if (32 + lane < u.n_pages) nxt = __ldg(idx + 32 + lane);
        }
        auto check_window = [&]() {
            const bool bad = win < 0 || static_cast<int64_t>(win) >= p.num_pages;
            if (__any_sync(0xffffffffu, bad) && lane == 0)
                record_status(p.status, p.epoch, kDeviceBadPage);
            win = bad ? 0 : win;  // an index outside the pool reads page 0
        };
        if (n_st > 0) check_window();
        const int n_slots = is_k ? kPKStages : kPVStages;
        uint64_t* full = is_k ? ctl.kfull : ctl.vfull;
        uint64_t* empty = is_k ? ctl.kempty : ctl.vempty;
        int* issued = is_k ? ctl.kissued : ctl.vissued;
        const CUtensorMap* map = is_k ? &tmap_k : &tmap_v;
        const int ca = p.layout == 0 ? u.hkv : 0;  // (d, A, B, page): NHD (d, head, token,
        const int cb = p.layout == 0 ? 0 : u.hkv;  // page), HND (d, token, head, page)
        bool ok = true;
        for (int s = 0; s < n_st; ++s) {
            const int slot = s % n_slots;
            const int pg0 = s * pps;
            const int npg = min(pps, u.n_pages - pg0);
            if (pg0 >= win_base + 32) {
                win = nxt;
                win_base += 32;
                nxt = win_base + 32 + lane < u.n_pages ? __ldg(idx + win_base + 32 + lane) : 0;
                check_window();
            }
            int okw = 1;
            if (lane == 0 && s >= n_slots)
                okw = mbar_wait_tc(&empty[slot], ((s / n_slots) + 1) & 1, flags, p.wait_ns) ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, okw, 0)) {
                ok = false;
                break;
            }
            if (lane == 0) {
                const uint32_t qbytes = is_k && s == 0 ? 2u * 128u * G * p.tile_tokens : 0u;
                mbar_arrive_expect_tx(&full[slot], npg * ps * kHeadDim * 2 + qbytes);
                if (qbytes) {
                    tma_load_3d(s_q, &tmap_q, &full[slot], 0, u.hkv * G, u.q_begin);
                    tma_load_3d(s_q + kPQHalf, &tmap_q, &full[slot], 64, u.hkv * G, u.q_begin);
                }
            }
            const int j = lane >> 1;
            const int page = __shfl_sync(0xffffffffu, win, (pg0 - win_base + j) & 31);
            if (lane < 2 * npg) {
                const uint32_t dst = (is_k ? ring_k(slot) : ring_v(slot)) + j * ps * 128 +
                                     ((lane & 1) ? kPHalf : 0);
                tma_load_4d(dst, map, &full[slot], (lane & 1) * 64, ca, cb, page);
            }
            if (lane == 0) issued[slot] += 1;
        }
        if (is_k && lane == 0 && usable) {
            // the device tables must be the ones the plan was made from
            const int b = u.b;
            const int64_t L = static_cast<int64_t>(p.indptr[b + 1] - p.indptr[b] - 1) * ps +
                              p.last_page_len[b];
            if ((p.qo_indptr != nullptr && p.qo_indptr[b] != u.qo_b) ||
                p.indptr[b] != u.page_base || L != u.kv_len)
                record_status(p.status, p.epoch, kDevicePlanMismatch);
        }
        if (!ok && lane == 0) {
            flags[0] = 1;
            record_status(p.status, p.epoch, kDeviceWaitTimeout);
        }
    } else if (warp == 4) {
        // ================================================ MMA warp
        if (lane == 0 && n_st > 0) {
            constexpr uint32_t kIdQK = umma_idesc(128, kNarrowStageTokens, 0);
            constexpr uint32_t kIdPV = umma_idesc(128, kHeadDim, 1);
            // Two kinds of work, each issued as soon as its inputs are ready:
            // the PV of stage gp (P written, V landed), checked first since it
            // frees a V slot and the score buffer of stage gp + 2, and the
            // score MMA of stage gq (K landed, its score buffer free). An idle
            // poll naps briefly so the softmax warps keep the issue slots.
            int gq = 0, gp = 0;
            bool ok = true;
            uint64_t idle_since = global_ns();
            while (gp < n_st) {
                bool progress = false;
                if (gp < gq && mbar_try_wait(&ctl.p_ready[gp & 1], (gp >> 1) & 1) &&
                    mbar_try_wait(&ctl.vfull[gp % kPVStages], (gp / kPVStages) & 1)) {
                    tc_fence_after();
                    // O += P V: 16 tokens a step = two 8-row groups (1024 B apart);
                    // the two 64-column halves of V are kPHalf apart
                    const uint32_t v0 = ring_v(gp % kPVStages);
                    for (int ks = 0; ks < kNarrowStageTokens / 16; ++ks) {
                        const uint64_t bd = umma_sdesc(v0 + ks * 2048, kPHalf, 1024);
                        umma_ts(t_o, t_s(gp & 1) + 8u * ks, bd, kIdPV,
                                (ks > 0 || gp > 0) ? 1u : 0u);
                    }
                    umma_commit(&ctl.vempty[gp % kPVStages]);
                    umma_commit(&ctl.o_ready[gp & 3]);
                    ++gp;
                    progress = true;
                }
                if (gq < n_st && gq < gp + 2 &&
                    mbar_try_wait(&ctl.kfull[gq % kPKStages], (gq / kPKStages) & 1)) {
                    tc_fence_after();
                    // S = Q K^T: K = 128 in steps of 16 (32 bytes of a 128-byte
                    // swizzled row; columns 64..127 in the other half)
                    const uint32_t k0 = ring_k(gq % kPKStages);
                    for (int ks = 0; ks < kHeadDim / 16; ++ks) {
                        const uint32_t h = static_cast<uint32_t>(ks >> 2), kk = ks & 3;
                        const uint64_t ad = umma_sdesc(s_q + h * kPQHalf + kk * 32, 16, 1024);
                        const uint64_t bd = umma_sdesc(k0 + h * kPHalf + kk * 32, 16, 1024);
                        umma_ss(t_s(gq & 1), ad, bd, kIdQK, ks > 0 ? 1u : 0u);
                    }
                    umma_commit(&ctl.s_ready[gq & 1]);
                    umma_commit(&ctl.kempty[gq % kPKStages]);  // K of the slot is consumed
                    ++gq;
                    progress = true;
                }
                if (progress) {
                    idle_since = global_ns();
                } else {
                    __nanosleep(32);
                }
                if (!progress && (flags[0] ||
                           global_ns() - idle_since > static_cast<uint64_t>(p.wait_ns))) {
                    ok = false;
                    break;
                }
            }
            if (!ok) {
                flags[0] = 1;
                record_status(p.status, p.epoch, kDeviceWaitTimeout);
            }
            // every MMA completes before the tensor memory is released
            umma_commit(&ctl.mma_done);
            mbar_wait_tc(&ctl.mma_done, 0, nullptr, kWaitTimeoutNs);
        }
        __syncwarp();
    } else {
        // ================================================ softmax warps
        // Thread r (< 128) owns row r = TMEM lane r; warp w reads lanes
        // [32w, 32w + 32). Every lane waits on each barrier itself; results
        // are AND-ed over the warp so the collective TMEM instructions see
        // one path.
        auto wait_all = [&](uint64_t* bar, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait_tc(bar, parity, flags, p.wait_ns));
        };
        const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
        const int r = threadIdx.x;  // 0 .. 127
        const int t = r / G, gi = r - (r / G) * G;
        const bool row_ok = r < G * p.tile_tokens && t < u.n_tok;
        const int pos = row_ok ? u.p0 + t : (1 << 30);  // padding rows see everything
        const float sc = p.scale_log2;
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int g = 0; g < n_st; ++g) {
            if (!wait_all(&ctl.s_ready[g & 1], (g >> 1) & 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[64];
            tmem_ld64(t_s(g & 1) + lane_off, sr);
            const int base = u.kv_begin + g * kNarrowStageTokens;
            const int nvalid = min(kNarrowStageTokens, u.kv_valid - g * kNarrowStageTokens);
            // A stage that ends at or before the tile's first position is seen
            // whole by every row (the same for the whole CTA): no mask, the
            // maximum is taken over the raw scores and the scale is folded
            // into the exponent's FMA. Otherwise scores are scaled and masked
            // first.
            const bool whole = nvalid == kNarrowStageTokens &&
                               base + kNarrowStageTokens - 1 <= u.p0 && sc > 0.f;
            float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            if (whole) {
#pragma unroll
                for (int j = 0; j < 64; j += 2)
                    mq[(j >> 1) & 3] = max3(mq[(j >> 1) & 3], __uint_as_float(sr[j]),
                                            __uint_as_float(sr[j + 1]));
            } else {
                const int lim = min(nvalid, pos - base + 1);  // visible columns of this row
#pragma unroll
                for (int j = 0; j < 64; ++j) {
                    const float x = j < lim ? __uint_as_float(sr[j]) * sc : -INFINITY;
                    sr[j] = __float_as_uint(x);
                    mq[j & 3] = fmaxf(mq[j & 3], x);
                }
            }
            float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
            if (whole) mx *= sc;
            float alpha = 1.f;
            bool rescale = false;
            if (g == 0) {
                m_ref = mx;
            } else if (mx > m_ref + 8.f) {
                alpha = fast_exp2(m_ref - mx);  // 0 while nothing was visible
                m_ref = mx;
                l *= alpha;
                rescale = true;
            }
            const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
            uint32_t pk[32];
            float lq[4] = {0.f, 0.f, 0.f, 0.f};
            if (whole) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    float x0, x1;
                    fma2(__uint_as_float(sr[2 * j]), __uint_as_float(sr[2 * j + 1]), sc, -m_use,
                         x0, x1);
                    const float p0 = fast_exp2(x0);
                    const float p1 = fast_exp2(x1);
                    add2(lq[(j & 1) * 2], lq[(j & 1) * 2 + 1], p0, p1);
                    pk[j] = pack_bf16x2(p0, p1);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float p0 = fast_exp2(__uint_as_float(sr[2 * j]) - m_use);
                    const float p1 = fast_exp2(__uint_as_float(sr[2 * j + 1]) - m_use);
                    lq[j & 3] += p0 + p1;
                    pk[j] = pack_bf16x2(p0, p1);
                }
            }
            l += (lq[0] + lq[1]) + (lq[2] + lq[3]);
            tmem_st32(t_s(g & 1) + lane_off, pk);
            tmem_wait_st();
            // PV(g - 1) must be done before O is rescaled; without a rescale
            // P(g) is published at once (PV(g) runs after PV(g - 1) anyway).
            // Four o_ready barriers keep every parity wait unambiguous: PV
            // (g + 3) cannot complete before this warp publishes P(g + 3),
            // and PV(g - 5) is known done from the wait of two stages ago.
            auto wait_pv = [&](int k) {
                return wait_all(&ctl.o_ready[k & 3], (k >> 2) & 1);
            };
            if (__any_sync(0xffffffffu, rescale)) {
                if (g > 0 && !wait_pv(g - 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int c0 = 0; c0 < kHeadDim; c0 += 64) {
                    uint32_t o[64];
                    tmem_ld64(t_o + lane_off + c0, o);
                    uint32_t w0[32], w1[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        w0[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                        w1[j] = __float_as_uint(__uint_as_float(o[32 + j]) * alpha);
                    }
                    tmem_st32(t_o + lane_off + c0, w0);
                    tmem_st32(t_o + lane_off + c0 + 32, w1);
                }
                tmem_wait_st();
            }
            const bool last = g == n_st - 1;
            if (last && nvalid < kNarrowStageTokens) {
                // zero V rows past the piece once its V landed (whole 128-byte
                // rows, so the swizzle does not matter); PV(g - 2) was issued
                // (QK(g) was), so this phase of vfull is the one for stage g
                if (!wait_all(&ctl.vfull[g % kPVStages], (g / kPVStages) & 1)) {
                    ok = false;
                    break;
                }
                uint8_t* v0 = sm + kPVOff + (g % kPVStages) * kPSlotBytes;
                const int n16 = (kNarrowStageTokens - nvalid) * 16;
                for (int i = r; i < n16; i += kPSoftmaxThreads) {
                    const int row = nvalid + (i >> 4), c = i & 15;
                    *reinterpret_cast<uint4*>(v0 + (c >> 3) * kPHalf + row * 128 + (c & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.p_ready[g & 1]);
            // follow the o_ready phases two stages behind, off the critical path
            if (g >= 2 && !wait_pv(g - 2)) {
                ok = false;
                break;
            }
            if (last) {
                // ---- epilogue: O / l, once PV(g) is done
                if (!wait_pv(g)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const bool seen = l > 0.f;  // a piece may lie wholly past a row's position
                const float inv = seen ? 1.f / l : 0.f;
                const float lse2 = seen ? m_ref + __log2f(l) : -INFINITY;
                const int hq = u.hkv * G + gi;
                for (int c0 = 0; c0 < kHeadDim; c0 += 64) {
                    uint32_t o[64];
                    tmem_ld64(t_o + lane_off + c0, o);
                    if (!row_ok) continue;
                    if (u.n_pieces == 1) {
                        uint16_t* dst =
                            p.out + (static_cast<size_t>(u.q_begin + t) * p.num_qo_heads + hq) *
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
                        const size_t grp =
                            static_cast<size_t>(u.state) +
                            static_cast<size_t>(t) * u.n_pieces + u.piece;
                        float* dst = p.part_o + (grp * G + gi) * kHeadDim + c0;
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
                    if (u.n_pieces == 1) {
                        if (p.lse != nullptr)
                            p.lse[static_cast<size_t>(u.q_begin + t) * p.num_qo_heads + hq] =
                                lse2 * kLn2;
                    } else {
                        const size_t grp =
                            static_cast<size_t>(u.state) +
                            static_cast<size_t>(t) * u.n_pieces + u.piece;
                        p.part_lse[grp * G + gi] = lse2;
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
        for (int s = 0; s < kPKStages; ++s)
            if (ctl.kissued[s] > 0)
                mbar_wait_tc(&ctl.kfull[s], (ctl.kissued[s] - 1) & 1, nullptr, kWaitTimeoutNs);
        for (int s = 0; s < kPVStages; ++s)
            if (ctl.vissued[s] > 0)
                mbar_wait_tc(&ctl.vfull[s], (ctl.vissued[s] - 1) & 1, nullptr, kWaitTimeoutNs);
    }
    if (warp == 4) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kPTmemCols)
                     : "memory");
    }
    // Started early behind another grid: that grid completes before this one
    // does, so a kernel that waits for this grid also sees the other's writes.
    if (p.wait_prior) asm volatile("griddepcontrol.wait;" ::: "memory");
}

cudaError_t ensure_narrow_attribute() {
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit != 0 && (done.load(std::memory_order_relaxed) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(paged_prefill_narrow_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kPSmemBytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_relaxed);
    return e;
}

}  // namespace

cudaError_t prefill_narrow_smem_bytes(int* bytes) {
    *bytes = kPSmemBytes;
    return cudaSuccess;
}

// Resident CTAs per SM from shared memory, threads and tensor-memory columns
// (the occupancy query answers 1 for kernels that use tcgen05).
cudaError_t prefill_narrow_occupancy(int* n) {
    cudaError_t e = ensure_narrow_attribute();
    if (e != cudaSuccess) return e;
    int dev = 0, smem_sm = 0, reserved = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
        cudaSuccess)
        return e;
    if ((e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) !=
        cudaSuccess)
        return e;
    const int by_smem = smem_sm / (kPSmemBytes + reserved);
    const int by_tmem = 512 / static_cast<int>(kPTmemCols);
    const int by_threads = 2048 / kPThreads;
    *n = max(1, min(by_smem, min(by_tmem, by_threads)));
    return cudaSuccess;
}

cudaError_t launch_prefill_narrow(const CUtensorMap& tk, const CUtensorMap& tv,
                                  const CUtensorMap& tq, const PrefillParams& p, int grid,
                                  cudaStream_t stream, bool early) {
    if (grid < 1 || (early && !p.wait_prior)) return cudaErrorInvalidConfiguration;
    cudaError_t e = ensure_narrow_attribute();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = kPSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = early ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, paged_prefill_narrow_kernel, tk, tv, tq, p);
}

}  // namespace oxd
