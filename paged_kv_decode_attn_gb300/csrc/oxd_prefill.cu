// Paged causal prefill for sm_103a on the 5th-generation tensor cores.
//
// Operation: "FlashInfer parity matrix" page, "Admitted attention matrix",
// row "Paged causal prefill" (BF16, D128, causal, NHD/HND pages through the
// same block tables as decode, split pieces with a caller-owned F32
// workspace), and "Domain coverage", "Prefill attention". Request b's query
// tokens are its last q_len_b cached tokens; query token i sits at position
// L_b - q_len_b + i and attends to cached tokens 0 .. that position.
//
// A tile is up to T = 256 / G consecutive query tokens of one request with
// the G query heads of one KV head each: 256 rows, row R = token R / G, head
// R % G, in two halves of 128 MMA rows. One CTA (one a SM: it holds all 512
// tensor-memory columns) runs one piece of a tile's cached-token range (a
// whole range, or one of the pieces of a split tile); eleven warps:
//   * K and V producers (warps 9, 10): per stage of 128 cached tokens one TMA
//     copy per (page, 64-column half) into a two-stage ring, laid out
//     [half][128 tokens][128 B] with the 128-byte swizzle; each stage serves
//     both halves of the tile;
//   * MMA warp (warp 8, issuing as a whole warp with one elected lane): per
//     half h, S_h = Q_h K^T (M = 128, N = 128, K = 128; Q_h and K in shared
//     memory) and O_h += P_h V (P_h from tensor memory; N = 128, K = 128) in a
//     fixed order, so the tensor core works on one half while the other's
//     softmax runs; a tile whose rows all fit in the first half gives it
//     both score buffers instead (QK(g + 1) runs during the softmax of g);
//   * softmax warpgroups (warps 0-3 for half 0, 4-7 for half 1): thread r
//     owns row r of its half (TMEM lane r). It first writes its query row
//     into shared memory. Per stage it loads the row's 128 scores and writes
//     P = 2^(s scale - m_ref) as bf16 pairs over the first 64 columns. A stage
//     that every row of the half sees whole (after the first) takes one pass
//     against the running reference m_ref, accepted when the row's sum shows
//     no term above 2^64; the first stage, the masked ones and a refused pass
//     take two (maximum, then P), masking the tokens past the row's position
//     and past the piece, and raise m_ref when the maximum exceeds it by more
//     than 2^8 (O_h is then rescaled in tensor memory: the score MMA's
//     completion means the previous PV is done). At the end the warpgroup
//     writes out/lse, or the F32 partial state of the piece.
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

constexpr int kPKStages = 2;     // K ring: a slot is free once both halves' score MMAs are done
constexpr int kPVStages = 2;     // V ring: a slot is free once both halves' PVs are done
constexpr int kPMmaWarp = 8;
constexpr int kPKWarp = 9;
constexpr int kPVWarp = 10;
constexpr int kPThreads = 11 * 32;
constexpr int kPHalf = kPrefillStageTokens * 128;  // one 64-column half of K or V: 16 KB
constexpr int kPSlotBytes = 2 * kPHalf;            // K or V of one stage: 32 KB
constexpr int kPQHalf = 128 * 128;                 // 64 columns of a half's 128 query rows
constexpr int kPQOff = 0;                          // Q of half h at 2 h kPQHalf: 64 KB
constexpr int kPKOff = kPQOff + 4 * kPQHalf;
constexpr int kPVOff = kPKOff + kPKStages * kPSlotBytes;
constexpr int kPCtlOff = kPVOff + kPVStages * kPSlotBytes;  // 192 KB of operands
// Tensor memory, 512 columns: per half h, O_h [128 h, 128 h + 128) and the
// scores (then P, bf16 pairs in the first 64 columns) S_h [256 + 128 h, +128).
constexpr uint32_t kPTmemCols = 512;
static_assert(kPKOff % 1024 == 0 && kPVOff % 1024 == 0 && kPSlotBytes % 1024 == 0,
              "swizzle atoms aligned");
static_assert(kPrefillStageTokens == 128, "score MMAs of N = 128, PV of K = 128");
static_assert(kPrefillRows == 2 * 128, "a tile is two 128-row halves");

struct PCtl {
    uint64_t kfull[kPKStages];
    uint64_t kempty[kPKStages];
    uint64_t vfull[kPVStages];
    uint64_t vempty[kPVStages];
    uint64_t q_ready[2];  // a half's query rows are in shared memory (one arrival a warp)
    uint64_t s_ready[2];  // QK_h(g) done: phase g of s_ready[h]
    uint64_t p_ready[2];  // P_h(g) written: phase g of p_ready[h] (one arrival a warp);
                          // a single-half tile's P(g): phase g / 2 of p_ready[g % 2]
    uint64_t o_done[2];   // the half's last PV done
    uint64_t pv_done;     // single-half tile: PV(g) done, phase g
    uint64_t vz;          // V rows past the piece zeroed (one arrival a warp)
    uint64_t mma_done;
    int kissued[kPKStages];
    int vissued[kPVStages];
    uint32_t tmem;
    int flags[4];  // [0] abort, [1] the unit is usable
};
// The dynamic shared memory starts 1024-byte aligned (checked in the kernel).
constexpr int kPSmemBytes = kPCtlOff + static_cast<int>(sizeof(PCtl));

// 32 lanes x 16 consecutive 32-bit columns, without the wait (see tmem_ld_wait16).
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait16(uint32_t (&r)[16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}

// Stages a half streams of a piece: its rows see cached tokens up to the
// position of its last query token.
__device__ __forceinline__ int half_stages(const PrefillUnit& u, int G, int h) {
    const int rows = u.n_tok * G;
    if (rows <= 128 * h) return 0;  // the half holds no row of the tile
    const int t_last = (min(rows, 128 * (h + 1)) - 1) / G;
    const int end = min(u.kv_begin + u.kv_valid, u.p0 + t_last + 1);
    return end > u.kv_begin ? (end - u.kv_begin + kPrefillStageTokens - 1) / kPrefillStageTokens
                            : 0;
}

__global__ void __launch_bounds__(kPThreads, 1)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v,
                         const __grid_constant__ PrefillParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* sm = smem_raw;
    PCtl& ctl = *reinterpret_cast<PCtl*>(sm + kPCtlOff);
    volatile int* flags = ctl.flags;
    const uint32_t s_base = smem_addr(sm);
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
        for (int h = 0; h < 2; ++h) {
            mbar_init(&ctl.q_ready[h], 4);
            mbar_init(&ctl.s_ready[h], 1);
            mbar_init(&ctl.p_ready[h], 4);
            mbar_init(&ctl.o_done[h], 1);
        }
        mbar_init(&ctl.pv_done, 1);
        mbar_init(&ctl.vz, 4);
        mbar_init(&ctl.mma_done, 1);
        flags[0] = 0;
        fence_mbar_init();
    }
    if (warp == kPMmaWarp) {
        asm volatile(
            "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                smem_addr(&ctl.tmem)),
            "r"(kPTmemCols)
            : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (warp == kPKWarp && lane == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
    }
    if (threadIdx.x == 0) {
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
                 u.kv_begin >= 0 && (u.kv_begin % kPrefillStageTokens) == 0 &&
                 static_cast<int64_t>(u.kv_begin % ps + u.kv_valid) <=
                     static_cast<int64_t>(u.n_pages) * ps &&
                 u.b >= 0 && u.b < p.batch && u.hkv >= 0 && u.hkv < p.num_kv_heads &&
                 u.n_tok >= 1 && u.n_tok <= T && u.n_tok * G <= kPrefillRows && u.q_begin >= 0 &&
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
        // The merge kernel, when the plan has one, may be scheduled now; it
        // waits for this grid to complete before it reads anything.
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl.tmem;
    auto t_o = [&](int h) { return tmem + 128u * static_cast<uint32_t>(h); };
    auto t_s = [&](int h) { return tmem + 256u + 128u * static_cast<uint32_t>(h); };
    auto s_q = [&](int h) { return s_base + kPQOff + 2u * kPQHalf * static_cast<uint32_t>(h); };
    const bool usable = flags[1] != 0;
    PrefillUnit u{};
    if (usable) u = p.units[blockIdx.x];
    const int n_st = usable ? (u.kv_valid + kPrefillStageTokens - 1) / kPrefillStageTokens : 0;
    const int nst_h[2] = {usable ? half_stages(u, G, 0) : 0, usable ? half_stages(u, G, 1) : 0};
    const int last_valid = n_st > 0 ? u.kv_valid - (n_st - 1) * kPrefillStageTokens : 0;
    // A tile whose rows all sit in the first half (half 1 streams nothing)
    // gives half 0 both score buffers: QK(g + 1) runs while the softmax of
    // stage g does.
    const bool single = nst_h[1] == 0;
    const bool need_vz = n_st > 0 && last_valid < kPrefillStageTokens;

    if (warp == kPKWarp || warp == kPVWarp) {
        // ================================================ producer warps
        // warp 9: K; warp 10: V. Lane 2j + c copies 64-column half c of page
        // j of the stage. Every stage serves both halves of the tile.
        const bool is_k = warp == kPKWarp;
        const int pps = kPrefillStageTokens / ps;  // pages per stage (divides 32)
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
                okw = mbar_wait(&empty[slot], ((s / n_slots) + 1) & 1, flags, p.wait_ns) ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, okw, 0)) {
                ok = false;
                break;
            }
            if (lane == 0) mbar_arrive_expect_tx(&full[slot], npg * ps * kHeadDim * 2);
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
    } else if (warp == kPMmaWarp) {
        // ================================================ MMA warp
        if (n_st > 0) {
            constexpr uint32_t kIdQK = umma_idesc(128, kPrefillStageTokens, 0);
            constexpr uint32_t kIdPV = umma_idesc(128, kHeadDim, 1);
            // Per half h: S_h = Q_h K^T (M = 128, N = 128 tokens, K = 128; both
            // operands in shared memory) and O_h += P_h V (P_h from tensor
            // memory; N = 128, K = 128 tokens). A fixed issue order with
            // blocking waits: QK_0(0), QK_1(0), then for each stage g
            // PV_0(g), QK_0(g + 1), PV_1(g), QK_1(g + 1). Within a half, QK_h(g + 1)
            // comes after PV_h(g) because it overwrites S_h, which holds P_h(g)
            // (MMAs from one thread run in issue order); across the halves the
            // tensor core works on one half while the other's softmax runs. A K
            // (V) slot is released once the last half that reads it has issued
            // its QK (PV) of that stage. Descriptors are a base plus constant
            // offsets (the start address field counts 16-byte units), so each
            // group of eight MMAs issues back to back. The whole warp runs this
            // loop (one elected lane issues), its waits agreed over the warp.
            const uint64_t qd0[2] = {umma_sdesc(s_q(0), 16, 1024), umma_sdesc(s_q(1), 16, 1024)};
            bool ok = true;
            auto wait = [&](uint64_t* bar, uint32_t parity) {
                ok = __all_sync(0xffffffffu, ok && mbar_wait_tc(bar, parity, flags, p.wait_ns));
                return ok;
            };
            auto issue_qk = [&](int h, int g, uint32_t sd) {
                // K = 128 in steps of 16: 32 bytes of a 128-byte swizzled row;
                // columns 64..127 in the other half
                const uint64_t kd0 = umma_sdesc(ring_k(g % kPKStages), 16, 1024);
#pragma unroll
                for (int ks = 0; ks < kHeadDim / 16; ++ks) {
                    const int c = ks >> 2, kk = ks & 3;
                    umma_ss_warp(sd, qd0[h] + static_cast<uint64_t>((c * kPQHalf + kk * 32) >> 4),
                                 kd0 + static_cast<uint64_t>((c * kPHalf + kk * 32) >> 4), kIdQK,
                                 ks > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int h, int g, uint32_t ps0) {
                // 16 tokens a step = two 8-row groups (1024 B apart); the two
                // 64-column halves of V are kPHalf apart
                const uint64_t vd0 = umma_sdesc(ring_v(g % kPVStages), kPHalf, 1024);
#pragma unroll
                for (int ks = 0; ks < kPrefillStageTokens / 16; ++ks)
                    umma_ts_warp(t_o(h), ps0 + 8u * ks, vd0 + static_cast<uint64_t>(ks * 2048 >> 4),
                                 kIdPV, (ks > 0 || g > 0) ? 1u : 0u);
            };
            if (single) {
                // Half 0 alone, scores in S_0 and S_1 by stage parity: QK(0),
                // QK(1), then per stage g PV(g) and QK(g + 2) into the buffer PV(g)
                // has just read P from.
                const int n = nst_h[0];
                for (int g = 0; g < min(n, 2) && ok; ++g) {
                    if (g == 0 && !wait(&ctl.q_ready[0], 0)) break;
                    if (!wait(&ctl.kfull[g % kPKStages], (g / kPKStages) & 1)) break;
                    tc_fence_after();
                    issue_qk(0, g, t_s(g & 1));
                    umma_commit_warp(&ctl.s_ready[g & 1]);
                    umma_commit_warp(&ctl.kempty[g % kPKStages]);
                }
                for (int g = 0; g < n && ok; ++g) {
                    // one barrier per score buffer: the softmax may publish
                    // P(g + 1) before this wait for P(g) has seen its phase
                    if (!wait(&ctl.p_ready[g & 1], (g >> 1) & 1)) break;
                    if (!wait(&ctl.vfull[g % kPVStages], (g / kPVStages) & 1)) break;
                    if (g == n_st - 1 && need_vz && !wait(&ctl.vz, 0)) break;
                    tc_fence_after();
                    issue_pv(0, g, t_s(g & 1));
                    umma_commit_warp(&ctl.pv_done);
                    umma_commit_warp(&ctl.vempty[g % kPVStages]);
                    if (g == n - 1) umma_commit_warp(&ctl.o_done[0]);
                    const int g2 = g + 2;
                    if (g2 < n) {
                        if (!wait(&ctl.kfull[g2 % kPKStages], (g2 / kPKStages) & 1)) break;
                        tc_fence_after();
                        issue_qk(0, g2, t_s(g2 & 1));
                        umma_commit_warp(&ctl.s_ready[g2 & 1]);
                        umma_commit_warp(&ctl.kempty[g2 % kPKStages]);
                    }
                }
            }
            const int n_max = single ? -1 : max(nst_h[0], nst_h[1]);
            for (int g = 0; g <= n_max && ok; ++g) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int gp = g - 1;  // the stage whose PV comes now
                    if (gp >= 0 && gp < nst_h[h]) {
                        if (!wait(&ctl.p_ready[h], gp & 1)) break;
                        if (h == 0 || gp >= nst_h[0]) {  // the first half to read V(gp)
                            if (!wait(&ctl.vfull[gp % kPVStages], (gp / kPVStages) & 1)) break;
                            if (gp == n_st - 1 && need_vz && !wait(&ctl.vz, 0)) break;
                        }
                        tc_fence_after();
                        issue_pv(h, gp, t_s(h));
                        if (gp == nst_h[h] - 1) umma_commit_warp(&ctl.o_done[h]);
                        if (h == 1 || gp >= nst_h[1])  // the last half to read V(gp)
                            umma_commit_warp(&ctl.vempty[gp % kPVStages]);
                    }
                    if (g < nst_h[h]) {
                        if (g == 0 && !wait(&ctl.q_ready[h], 0)) break;
                        if ((h == 0 || g >= nst_h[0]) &&
                            !wait(&ctl.kfull[g % kPKStages], (g / kPKStages) & 1))
                            break;
                        tc_fence_after();
                        issue_qk(h, g, t_s(h));
                        umma_commit_warp(&ctl.s_ready[h]);
                        if (h == 1 || g >= nst_h[1])  // the last half to read K(g)
                            umma_commit_warp(&ctl.kempty[g % kPKStages]);
                    }
                }
            }
            if (!ok && lane == 0) {
                flags[0] = 1;
                record_status(p.status, p.epoch, kDeviceWaitTimeout);
            }
            // every MMA completes before the tensor memory is released
            umma_commit_warp(&ctl.mma_done);
            mbar_wait(&ctl.mma_done, 0, nullptr, kWaitTimeoutNs);
        }
        __syncwarp();
    } else {
        // ================================================ softmax warpgroups
        // Warpgroup h (warps 4h .. 4h + 3) owns half h of the tile; thread r of
        // the warpgroup owns row 128 h + r of the tile, TMEM lane r (warp w
        // reads lanes [32 (w % 4), +32)). Every lane waits on each barrier
        // itself; results are AND-ed over the warp so the collective TMEM
        // instructions see one path.
        auto wait_all = [&](uint64_t* bar, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity, flags, p.wait_ns));
        };
        const int h = warp >> 2;
        const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
        const int r = threadIdx.x & 127;
        const int R = 128 * h + r;  // row of the tile: token R / G, head R % G
        const int t = R / G, gi = R - (R / G) * G;
        const bool row_ok = usable && t < u.n_tok;
        const int pos = row_ok ? u.p0 + t : (1 << 30);  // padding rows see everything
        const int nst = nst_h[h];
        // the half's query rows into shared memory (once; zeros past the
        // tile), laid out as the score MMA's A operand: two 64-column halves
        // of [128 rows][128 B] with the 128-byte swizzle (16-byte chunk j of
        // row r at chunk j ^ (r % 8))
        if (nst > 0) {
            const uint4* src = reinterpret_cast<const uint4*>(
                p.q + (static_cast<size_t>(u.q_begin + (row_ok ? t : 0)) * p.num_qo_heads +
                       u.hkv * G + (row_ok ? gi : 0)) *
                          kHeadDim);
            uint8_t* qs = sm + kPQOff + 2 * kPQHalf * h + r * 128;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint4 w = row_ok ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(qs + (i >> 3) * kPQHalf + (((i & 7) ^ (r & 7)) << 4)) = w;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.q_ready[h]);
        }
        // the half's first row position: a stage ending at or before it is
        // seen whole by every row of the half
        const int p_first = usable ? u.p0 + (128 * h) / G : 0;
        // the half with the tile's last rows streams every stage of the piece;
        // its warps zero V rows past the piece
        const bool zeroes = need_vz && h == (usable && u.n_tok * G > 128 ? 1 : 0);
        const float sc = p.scale_log2;
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int g = 0; g < nst; ++g) {
            // the stage's score buffer: S_h, or S_(g % 2) for a single-half tile
            const int sb = single ? (g & 1) : h;
            const uint32_t ts = t_s(sb);
            if (!wait_all(&ctl.s_ready[sb], single ? (g >> 1) & 1 : g & 1)) {
                ok = false;
                break;
            }
            // s_ready(g) also means every MMA issued before QK_h(g) is done:
            // PV_h(g - 1) among them with two halves (O_h is up to date), and
            // PV(g - 2) for a single-half tile (its P was in this buffer)
            tc_fence_after();
            const int base = u.kv_begin + g * kPrefillStageTokens;
            const int nvalid = min(kPrefillStageTokens, u.kv_valid - g * kPrefillStageTokens);
            // A stage that ends at or before the half's first position is seen
            // whole by every row (the same for the whole warpgroup): no mask,
            // the maximum is taken over the raw scores and the scale is folded
            // into the exponent's FMA. Otherwise scores are scaled and masked.
            const bool whole = nvalid == kPrefillStageTokens &&
                               base + kPrefillStageTokens - 1 <= p_first && sc > 0.f;
            const int lim = min(nvalid, pos - base + 1);  // visible columns of this row
            float lq[4] = {0.f, 0.f, 0.f, 0.f};
            bool rescale = false;
            float alpha = 1.f;
            bool done = false;
            if (whole && g > 0) {
                // One pass against the running reference m_ref (no maximum): P =
                // 2^(s sc - m_ref) for 16 columns at a time (the next 16 loading
                // meanwhile), kept in registers until the row's sum shows that no
                // term exceeds 2^64 (nor is infinite); then P is bf16 and O and l
                // are F32 well inside their range. Otherwise the two passes below
                // run (the scores are still in tensor memory). The reference may
                // lag the row's maximum: every term carries the same factor
                // 2^(m - m_ref), which the final O / l cancels.
                uint32_t pk[64];
                uint32_t a[16], b[16];
                auto chunk = [&](const uint32_t (&x)[16], int i) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        float x0, x1;
                        fma2(__uint_as_float(x[2 * j]), __uint_as_float(x[2 * j + 1]), sc, -m_ref,
                             x0, x1);
                        const float p0 = fast_exp2(x0);
                        const float p1 = fast_exp2(x1);
                        add2(lq[(j & 1) * 2], lq[(j & 1) * 2 + 1], p0, p1);
                        pk[8 * i + j] = pack_bf16x2(p0, p1);
                    }
                };
                tmem_ld16_async(ts + lane_off, a);
                tmem_ld_wait16(a);
#pragma unroll
                for (int i = 0; i < 8; i += 2) {
                    tmem_ld16_async(ts + lane_off + 16 * (i + 1), b);
                    chunk(a, i);
                    tmem_ld_wait16(b);
                    if (i + 2 < 8) tmem_ld16_async(ts + lane_off + 16 * (i + 2), a);
                    chunk(b, i + 1);
                    if (i + 2 < 8) tmem_ld_wait16(a);
                }
                const float ltot = (lq[0] + lq[1]) + (lq[2] + lq[3]);
                if (!__any_sync(0xffffffffu, !(ltot <= 0x1p64f))) {
                    uint32_t (&p0)[32] = *reinterpret_cast<uint32_t (*)[32]>(&pk[0]);
                    uint32_t (&p1)[32] = *reinterpret_cast<uint32_t (*)[32]>(&pk[32]);
                    tmem_st32(ts + lane_off, p0);
                    tmem_st32(ts + lane_off + 32, p1);
                    done = true;
                } else {
                    lq[0] = lq[1] = lq[2] = lq[3] = 0.f;
                }
            }
            if (!done) {
                // Scores of tokens 0..63 stay in registers; those of 64..127 are
                // read twice (for the maximum, then for P), which keeps the
                // thread within its register share. P (bf16 pairs) goes to
                // columns 0..63, over scores already read.
                uint32_t s0[64];
                tmem_ld64(ts + lane_off, s0);
                float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                if (whole) {
#pragma unroll
                    for (int j = 0; j < 64; j += 2)
                        mq[(j >> 1) & 3] = max3(mq[(j >> 1) & 3], __uint_as_float(s0[j]),
                                                __uint_as_float(s0[j + 1]));
                } else {
#pragma unroll
                    for (int j = 0; j < 64; ++j) {
                        const float x = j < lim ? __uint_as_float(s0[j]) * sc : -INFINITY;
                        s0[j] = __float_as_uint(x);
                        mq[j & 3] = fmaxf(mq[j & 3], x);
                    }
                }
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t s1[32];
                    tmem_ld32(ts + lane_off + 64 + 32 * c, s1);
                    if (whole) {
#pragma unroll
                        for (int j = 0; j < 32; j += 2)
                            mq[(j >> 1) & 3] = max3(mq[(j >> 1) & 3], __uint_as_float(s1[j]),
                                                    __uint_as_float(s1[j + 1]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            mq[j & 3] = fmaxf(mq[j & 3], 64 + 32 * c + j < lim
                                                             ? __uint_as_float(s1[j]) * sc
                                                             : -INFINITY);
                    }
                }
                float mx = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
                if (whole) mx *= sc;
                if (g == 0) {
                    m_ref = mx;
                } else if (mx > m_ref + 8.f) {
                    alpha = fast_exp2(m_ref - mx);  // 0 while nothing was visible
                    m_ref = mx;
                    l *= alpha;
                    rescale = true;
                }
                const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
                {
                    uint32_t pk[32];
                    if (whole) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            float x0, x1;
                            fma2(__uint_as_float(s0[2 * j]), __uint_as_float(s0[2 * j + 1]), sc,
                                 -m_use, x0, x1);
                            const float p0 = fast_exp2(x0);
                            const float p1 = fast_exp2(x1);
                            add2(lq[(j & 1) * 2], lq[(j & 1) * 2 + 1], p0, p1);
                            pk[j] = pack_bf16x2(p0, p1);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const float p0 = fast_exp2(__uint_as_float(s0[2 * j]) - m_use);
                            const float p1 = fast_exp2(__uint_as_float(s0[2 * j + 1]) - m_use);
                            lq[j & 3] += p0 + p1;
                            pk[j] = pack_bf16x2(p0, p1);
                        }
                    }
                    tmem_st32(ts + lane_off, pk);
                }
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t s1[32], pk[16];
                    tmem_ld32(ts + lane_off + 64 + 32 * c, s1);
                    if (whole) {
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            float x0, x1;
                            fma2(__uint_as_float(s1[2 * j]), __uint_as_float(s1[2 * j + 1]), sc,
                                 -m_use, x0, x1);
                            const float p0 = fast_exp2(x0);
                            const float p1 = fast_exp2(x1);
                            add2(lq[(j & 1) * 2], lq[(j & 1) * 2 + 1], p0, p1);
                            pk[j] = pack_bf16x2(p0, p1);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int t0 = 64 + 32 * c + 2 * j;
                            const float x0 = t0 < lim ? __uint_as_float(s1[2 * j]) * sc : -INFINITY;
                            const float x1 =
                                t0 + 1 < lim ? __uint_as_float(s1[2 * j + 1]) * sc : -INFINITY;
                            const float p0 = fast_exp2(x0 - m_use);
                            const float p1 = fast_exp2(x1 - m_use);
                            lq[j & 3] += p0 + p1;
                            pk[j] = pack_bf16x2(p0, p1);
                        }
                    }
                    tmem_st16(ts + lane_off + 32 + 16 * c, pk);
                }
            }
            l += (lq[0] + lq[1]) + (lq[2] + lq[3]);
            if (__any_sync(0xffffffffu, rescale)) {
                // O_h holds PV_h through stage g - 1: done (see above), or
                // waited for here for a single-half tile
                if (single && !wait_all(&ctl.pv_done, (g - 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int c0 = 0; c0 < kHeadDim; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(t_o(h) + lane_off + c0, o);
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
                    tmem_st32(t_o(h) + lane_off + c0, o);
                }
            }
            tmem_wait_st();
            const bool last = g == nst - 1;
            if (last && zeroes) {
                // zero V rows past the piece once its V landed (whole 128-byte
                // rows, so the swizzle does not matter); V(g - 2), the slot's
                // previous stage, has been read (PV(g - 2) is done), so this
                // phase of vfull is the one for stage g
                if (!wait_all(&ctl.vfull[g % kPVStages], (g / kPVStages) & 1)) {
                    ok = false;
                    break;
                }
                uint8_t* v0 = sm + kPVOff + (g % kPVStages) * kPSlotBytes;
                const int n16 = (kPrefillStageTokens - nvalid) * 16;
                for (int i = r; i < n16; i += 128) {
                    const int row = nvalid + (i >> 4), c = i & 15;
                    *reinterpret_cast<uint4*>(v0 + (c >> 3) * kPHalf + row * 128 + (c & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl.vz);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl.p_ready[sb]);
        }
        // ---- epilogue: O / l once the half's last PV is done; padding rows
        // take part in the collective loads. A piece wholly past the half's
        // rows leaves them an empty state (a split tile's merge weighs it 0).
        if (ok && nst > 0 && !wait_all(&ctl.o_done[h], 0)) ok = false;
        if (ok && (nst > 0 || (row_ok && u.n_pieces > 1))) {
            tc_fence_after();
            const bool seen = l > 0.f;  // a piece may lie wholly past a row's position
            const float inv = seen ? 1.f / l : 0.f;
            const float lse2 = seen ? m_ref + __log2f(l) : -INFINITY;
            const int hq = u.hkv * G + gi;
            for (int c0 = 0; c0 < kHeadDim; c0 += 64) {
                uint32_t o[64];
                if (nst > 0) {
                    tmem_ld64(t_o(h) + lane_off + c0, o);
                } else {
#pragma unroll
                    for (int j = 0; j < 64; ++j) o[j] = 0u;
                }
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
                    const size_t grp = static_cast<size_t>(u.state) +
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
                    const size_t grp = static_cast<size_t>(u.state) +
                                       static_cast<size_t>(t) * u.n_pieces + u.piece;
                    p.part_lse[grp * G + gi] = lse2;
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
                mbar_wait(&ctl.kfull[s], (ctl.kissued[s] - 1) & 1, nullptr, kWaitTimeoutNs);
        for (int s = 0; s < kPVStages; ++s)
            if (ctl.vissued[s] > 0)
                mbar_wait(&ctl.vfull[s], (ctl.vissued[s] - 1) & 1, nullptr, kWaitTimeoutNs);
    }
    if (warp == kPMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kPTmemCols)
                     : "memory");
    }
    // Started early behind another grid: that grid completes before this one
    // does, so a kernel that waits for this grid also sees the other's writes.
    if (p.wait_prior) asm volatile("griddepcontrol.wait;" ::: "memory");
}

cudaError_t ensure_prefill_attribute() {
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit != 0 && (done.load(std::memory_order_relaxed) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(paged_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kPSmemBytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_relaxed);
    return e;
}

}  // namespace

cudaError_t prefill_smem_bytes(int* bytes) {
    *bytes = kPSmemBytes;
    return cudaSuccess;
}

// Resident CTAs per SM from shared memory, threads and tensor-memory columns
// (the occupancy query answers 1 for kernels that use tcgen05).
cudaError_t prefill_occupancy(int* n) {
    cudaError_t e = ensure_prefill_attribute();
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
    *n = max(1, min(by_smem, min(by_tmem, by_threads)));  // one CTA a SM
    return cudaSuccess;
}

cudaError_t launch_prefill(const CUtensorMap& tk, const CUtensorMap& tv, const PrefillParams& p,
                           int grid, cudaStream_t stream, bool early) {
    if (grid < 1 || (early && !p.wait_prior)) return cudaErrorInvalidConfiguration;
    cudaError_t e = ensure_prefill_attribute();
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
    return cudaLaunchKernelEx(&cfg, paged_prefill_kernel, tk, tv, p);
}

}  // namespace oxd
