// Paged-KV decode attention kernels for sm_103a.
//
// Operation: "FlashInfer parity matrix" page, "Admitted attention matrix",
// row "Paged batch decode" (direct kernel for MHA, eight-warp token-parallel
// kernel for MQA/GQA), with the F32 online softmax every attention row there
// fixes, and the split partitions + F32 partial workspace + merge of the
// "Single decode split-K" row.
//
// Persistent, warp-specialised CTAs (a few per SM). The planner lays the
// page streams of all (request, KV head) pairs end to end and cuts them into
// one equal share per CTA; a share is a few work units, each a run of
// consecutive pages of one request for one KV head:
//   * the producer warp reads the next unit's entry while the current one is
//     still streaming, reads its page indices 32 at a time (coalesced), checks them
//     against the pool, and fills a ring of shared-memory stages: one TMA
//     tensor copy per (page, 64-column half) for K and for V, plus, on a
//     unit's first stage, a bulk copy of the group's G query rows; every
//     stage carries a small record (request, head, stage index, output slot)
//     and is guarded by a "full" and an "empty" mbarrier;
//   * consumer warps split each stage token-parallel, 16 tokens per warp, and
//     keep their own running max, denominator and F32 accumulator; for
//     grouped heads (G >= 3) the group's query rows are the A operand of
//     mma.sync m16n8k16 for Q K^T and the bf16-rounded softmax weights the A
//     operand of P V, so one K/V read serves all G heads; for G <= 2 the dot
//     products run on CUDA cores;
//   * after a unit's last stage the consumers merge their states through the
//     stage's own buffer and write the bf16 output and LSE, or, for a split
//     request, an F32 partial state that the merge kernel (launched right
//     behind this one) combines;
//   * a small batch may instead be launched as thread-block clusters, one
//     stream per cluster and one piece per CTA: each piece's state goes to
//     the shared memory of the cluster's first CTA, which merges them.
// The work list travels in the kernel's parameter buffer when it fits, and
// the device status word carries the run's epoch, so a run enqueues nothing
// but its kernels.
// Every mbarrier wait gives up after about one second:
// it records OXD_DEVICE_WAIT_TIMEOUT, all warps leave (the consumer warps
// decide together through a barrier reduction, so no named barrier can be
// left waiting), the copies already issued are drained, and the CTA returns.
#include <cuda_bf16.h>

#include <atomic>
#include <type_traits>

#include "oxd_internal.h"
#include "oxd_merge_row.cuh"
#include "oxd_ptx.cuh"

namespace oxd {
namespace {

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ float lds_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// D = A * B + D, m16n8k16, bf16 inputs, f32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Named barrier 1 among the consumer warps (the producer warp never uses it).
__device__ __forceinline__ void consumer_sync(int nthreads) {
    asm volatile("barrier.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// Same barrier, returning the AND of every participant's `v`.
__device__ __forceinline__ bool consumer_all(int nthreads, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "barrier.red.and.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(nthreads)
        : "memory");
    return r != 0;
}


// ------------------------------------------------------------------ tile addressing
//
// A stage holds K then V for kStageTokens tokens. Each is a sequence of TMA
// boxes of R = page_size rows (one page of one KV head); a box is two
// [R][64] bf16 halves (d < 64, then d >= 64), 128-byte rows, written by TMA
// with the 128-byte swizzle: 16-byte chunk cc of row r sits at chunk
// cc ^ (r % 8). Every half starts on a 1024-byte boundary (R is a multiple
// of 8), so the swizzle phase is r % 8 = t % 8.
//
// Byte offset of 16-byte chunk c (0..15, i.e. d = 8c..8c+7) of token t:
//   (t / R) * R * 256 + (c / 8) * R * 128 + (t % R) * 128 + ((c % 8) ^ (t % 8)) * 16
// and (t / R) * R * 256 + (t % R) * 128 = t * 256 - (t % R) * 128.
struct RowAddr {
    uint32_t base;  // tile base + t * 256 - (t % R) * 128
    uint32_t xr;    // t % 8
};

__device__ __forceinline__ RowAddr row_addr(uint32_t tile, int t, int rmask) {
    const int r = t & rmask;
    return {tile + static_cast<uint32_t>(t * 256 - r * 128), static_cast<uint32_t>(t & 7)};
}

__device__ __forceinline__ uint32_t chunk_addr(const RowAddr& ra, int c, int half_bytes) {
    return ra.base + static_cast<uint32_t>((c >> 3) * half_bytes) +
           ((static_cast<uint32_t>(c & 7) ^ ra.xr) << 4);
}

// Epilogue scratch: per consumer warp slice, a [16][128] f32 block of its
// accumulator rows, stored in the stage buffer the unit finished with. Column
// groups of 8 are XOR-swizzled by row % 8 to spread the banks.
__device__ __forceinline__ int dump_col(int row, int col) { return col ^ ((row & 7) << 3); }

// ------------------------------------------------------------------ configuration

template <int kMtiles_, bool kHiRows_, int kSlices_, int kStages_, bool kMma_, int kFmaGroup_>
struct Cfg {
    static constexpr int kMtiles = kMtiles_;       // 16-row query tiles (mma)
    static constexpr bool kHiRows = kHiRows_;      // rows 8..15 of a tile in use
    static constexpr int kSlices = kSlices_;       // token slices per stage
    static constexpr int kStages = kStages_;
    static constexpr bool kMma = kMma_;
    static constexpr int kFmaGroup = kFmaGroup_;   // G of the CUDA-core variant
    static constexpr int kConsumerWarps = kMma ? kSlices * kMtiles : kSlices;
    // Register budget: two CTAs of five warps share an SM, so one of its four
    // register files holds three warps, which fits at most 168 registers a
    // thread. The 16-row tensor-core and the CUDA-core variants run faster
    // with all 168; the 8-row variant runs faster with the compiler's own
    // choice under the launch bound.
    static constexpr bool kRegs168 = !kMma || kHiRows;
    static constexpr int kConsumerThreads = kConsumerWarps * 32;
    static constexpr int kThreads = kConsumerThreads + 32;
    static constexpr int kStageTokens = kSlices * kSliceTokens;
    static constexpr int kStageBytes = kStageTokens * kHeadDim * 2 * 2;  // K and V
    static constexpr int kQRows = kMma ? (kHiRows ? 16 * kMtiles : 8) : kFmaGroup;
    static constexpr int kQBytes = kQRows * kHeadDim * 2;
    static_assert(kSlices * 16 * kHeadDim * 4 <= kStageBytes, "epilogue scratch fits a stage");
    // ring | q[kStages] | rec[kStages] | full, empty, cluster | issued | flags | red_m | red_l
    static constexpr int kQOffset = kStages * kStageBytes;
    static constexpr int kRecOffset = kQOffset + kStages * kQBytes;
    static constexpr int kBarOffset = kRecOffset + kStages * 32;
    static constexpr int kIssuedOffset = kBarOffset + (2 * kStages + 1) * 8;
    static constexpr int kFlagOffset = (kIssuedOffset + kStages * 4 + 15) / 16 * 16;
    static constexpr int kRedOffset = kFlagOffset + 16;
    static constexpr int kSmemBytes = 1024 /* alignment slack */ + kRedOffset +
                                      2 * kConsumerWarps * 16 * 4;
    // Cluster launches add a region for the pieces' final states, filled by
    // the cluster's CTAs in rank 0: [kMaxClusterCtas][kQRows][128] f32 values,
    // then [kMaxClusterCtas][kQRows] f32 log2-sums.
    static constexpr int kClusterOff = (kSmemBytes - 1024 + 15) / 16 * 16;
    static constexpr int kClusterOBytes = kMaxClusterCtas * kQRows * kHeadDim * 4;
    static constexpr int kSmemBytesCluster =
        1024 + kClusterOff + kClusterOBytes + kMaxClusterCtas * kQRows * 4;
    // alignment each region's accesses need (the base is 1024-aligned)
    static_assert(kStageBytes % 1024 == 0, "stages keep the 128-byte swizzle atoms aligned");
    static_assert(kQOffset % 128 == 0 && kQBytes % 128 == 0, "query rows: bulk copy, ldmatrix");
    static_assert(kRecOffset % 16 == 0, "stage records");
    static_assert(kBarOffset % 8 == 0, "mbarriers");
    static_assert(kFlagOffset % 16 == 0 && kRedOffset % 16 == 0, "flags, reductions");
};

using CfgFmaG1 = Cfg<1, false, 4, 3, false, 1>;
using CfgFmaG2 = Cfg<1, false, 4, 3, false, 2>;
using CfgMma8 = Cfg<1, false, 4, 3, true, 0>;
using CfgMma16 = Cfg<1, true, 4, 3, true, 0>;

// Configuration of a cluster launch. A cluster's pieces are short (a few
// stages each), so the 8-row tensor-core variant gives up a ring stage to
// hold the eight pieces' states of its up to 8 rows in rank 0 (about 103 KB
// a CTA, still two a SM); the CUDA-core variants keep theirs.
template <class C> struct ClusterCfg { using type = C; };
template <> struct ClusterCfg<CfgMma8> { using type = Cfg<1, false, 4, 2, true, 0>; };

// What the producer tells the consumers about each stage it fills.
struct StageRec {
    int b, hkv, valid, n_stages, s, slot, row0, nrows;  // query rows [row0, row0+nrows) of the group
};

// ------------------------------------------------------------------ consumers

// Tensor-core consumer: one warp owns query rows [16*mt, 16*mt + 16) of the
// group and one 16-token slice of every stage.
template <class C>
struct MmaConsumer {
    uint32_t qa[8][4];   // A fragments of the query rows, one per 16-wide k step
    float m[2];          // running max (log2 domain) of rows g, g + 8
    float l[2];          // running denominator (this thread's columns)
    float acc[16][4];    // output accumulator, 16 n-tiles of 8 columns

    // q rows come from the stage's query buffer (row r at qbuf + 256 r).
    __device__ __forceinline__ void init(uint32_t qbuf, int G, int mt, int lane) {
        const int g = lane >> 2, tq = lane & 3;
        const int r0 = mt * 16 + g, r1 = r0 + 8;
        const bool v0 = r0 < G, v1 = C::kHiRows && r1 < G;
        const uint32_t a0 = qbuf + r0 * 256 + tq * 4;
        const uint32_t a1 = qbuf + r1 * 256 + tq * 4;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            qa[ks][0] = v0 ? lds32(a0 + ks * 32) : 0u;
            qa[ks][1] = v1 ? lds32(a1 + ks * 32) : 0u;
            qa[ks][2] = v0 ? lds32(a0 + ks * 32 + 16) : 0u;
            qa[ks][3] = v1 ? lds32(a1 + ks * 32 + 16) : 0u;
        }
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.f;
#pragma unroll
        for (int n = 0; n < 16; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    }

    // Tokens [u0, u0 + 16) of the unit sit at rows t0.. of the stage tiles.
    __device__ __forceinline__ void consume(uint32_t tk, uint32_t tv, int t0, int u0, int valid,
                                            int rmask, int half_bytes, float scale_log2,
                                            int lane) {
        const int mi = lane >> 3, ri = lane & 7;
        // ---- S = Q K^T for 16 tokens: two n-tiles of 8 tokens
        // Even and odd k steps accumulate separately: two independent mma
        // chains per n-tile halve the dependent latency; summed afterwards.
        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        float s2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        const RowAddr rk = row_addr(tk, t0 + ((mi >> 1) << 3) + ri, rmask);
#pragma unroll
        for (int ks = 0; ks < 8; ks += 2) {
            uint32_t b0, b1, b2, b3, c0, c1, c2, c3;
            ldsm_x4(chunk_addr(rk, 2 * ks + (mi & 1), half_bytes), b0, b1, b2, b3);
            ldsm_x4(chunk_addr(rk, 2 * ks + 2 + (mi & 1), half_bytes), c0, c1, c2, c3);
            mma_bf16(s[0], qa[ks], b0, b1);
            mma_bf16(s[1], qa[ks], b2, b3);
            mma_bf16(s2[0], qa[ks + 1], c0, c1);
            mma_bf16(s2[1], qa[ks + 1], c2, c3);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            s[0][e] += s2[0][e];
            s[1][e] += s2[1][e];
        }
        // ---- online softmax in the log2 domain
        const int tq = lane & 3;
        const bool partial = u0 + kSliceTokens > valid;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int tok = u0 + nt * 8 + 2 * tq + (e & 1);
                const float x = s[nt][e] * scale_log2;
                s[nt][e] = (partial && tok >= valid) ? -INFINITY : x;
            }
        }
        float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        const float mn0 = fmaxf(m[0], mx0);
        const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
        const float al0 = fast_exp2(m[0] - mu0);
        m[0] = mn0;
        s[0][0] = fast_exp2(s[0][0] - mu0);
        s[0][1] = fast_exp2(s[0][1] - mu0);
        s[1][0] = fast_exp2(s[1][0] - mu0);
        s[1][1] = fast_exp2(s[1][1] - mu0);
        l[0] = l[0] * al0 + ((s[0][0] + s[0][1]) + (s[1][0] + s[1][1]));
        float al1 = 1.f;
        if constexpr (C::kHiRows) {
            float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float mn1 = fmaxf(m[1], mx1);
            const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
            al1 = fast_exp2(m[1] - mu1);
            m[1] = mn1;
            s[0][2] = fast_exp2(s[0][2] - mu1);
            s[0][3] = fast_exp2(s[0][3] - mu1);
            s[1][2] = fast_exp2(s[1][2] - mu1);
            s[1][3] = fast_exp2(s[1][3] - mu1);
            l[1] = l[1] * al1 + ((s[0][2] + s[0][3]) + (s[1][2] + s[1][3]));
        } else {
            s[0][2] = s[0][3] = s[1][2] = s[1][3] = 0.f;
        }
        // The accumulator only needs rescaling when some row's running max
        // rose (alpha < 1); after the first tiles that is rare.
        if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                acc[n][0] *= al0;
                acc[n][1] *= al0;
                if constexpr (C::kHiRows) {
                    acc[n][2] *= al1;
                    acc[n][3] *= al1;
                }
            }
        }
        // ---- O += P V: P (bf16) is the A operand, built from the S fragments
        uint32_t pa[4];
        pa[0] = pack_bf16x2(s[0][0], s[0][1]);
        pa[1] = pack_bf16x2(s[0][2], s[0][3]);
        pa[2] = pack_bf16x2(s[1][0], s[1][1]);
        pa[3] = pack_bf16x2(s[1][2], s[1][3]);
        // V rows of tokens past `valid` may hold anything (even NaN): zero the
        // corresponding halves of the B fragments, not just their weights.
        uint32_t keep0 = 0xffffffffu, keep1 = 0xffffffffu;
        if (partial) {
            const int k0 = u0 + 2 * tq;
            keep0 = (k0 < valid ? 0x0000ffffu : 0u) | (k0 + 1 < valid ? 0xffff0000u : 0u);
            keep1 = (k0 + 8 < valid ? 0x0000ffffu : 0u) | (k0 + 9 < valid ? 0xffff0000u : 0u);
        }
        const RowAddr rv = row_addr(tv, t0 + ((mi & 1) << 3) + ri, rmask);
#pragma unroll
        for (int np = 0; np < 8; ++np) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_trans(chunk_addr(rv, 2 * np + (mi >> 1), half_bytes), b0, b1, b2, b3);
            mma_bf16(acc[2 * np], pa, b0 & keep0, b1 & keep1);
            mma_bf16(acc[2 * np + 1], pa, b2 & keep0, b3 & keep1);
        }
    }

    // Raw state of this warp's 16 rows: red_m/red_l [slice][16] and the
    // accumulator into dump + slice * 16 * 128 (rows swizzled by dump_col).
    __device__ __forceinline__ void dump(float* red_m, float* red_l, float* dump, int slice,
                                         int lane) {
        const int g = lane >> 2, tq = lane & 3;
        float l0 = l[0], l1 = l[1];
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
        if (tq == 0) {
            red_m[slice * 16 + g] = m[0];
            red_l[slice * 16 + g] = l0;
            red_m[slice * 16 + g + 8] = C::kHiRows ? m[1] : -INFINITY;
            red_l[slice * 16 + g + 8] = C::kHiRows ? l1 : 0.f;
        }
        float* base = dump + slice * 16 * kHeadDim;
#pragma unroll
        for (int n = 0; n < 16; ++n) {
            const int col = n * 8 + 2 * tq;
            *reinterpret_cast<float2*>(base + g * kHeadDim + dump_col(g, col)) =
                make_float2(acc[n][0], acc[n][1]);
            if constexpr (C::kHiRows)
                *reinterpret_cast<float2*>(base + (g + 8) * kHeadDim + dump_col(g + 8, col)) =
                    make_float2(acc[n][2], acc[n][3]);
        }
    }
};

// CUDA-core consumer for G <= 2: lane = (token parity, 16-byte chunk of D).
template <class C>
struct FmaConsumer {
    static constexpr int G = C::kFmaGroup;
    float qf[G][8];
    float m[G];
    float l[G];
    float acc[G][8];

    __device__ __forceinline__ void init(uint32_t qbuf, int /*G*/, int /*mt*/, int lane) {
        const int c = lane & 15;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const uint4 raw = lds128(qbuf + g * 256 + c * 16);
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                qf[g][2 * j] = bf16_lo(w[j]);
                qf[g][2 * j + 1] = bf16_hi(w[j]);
            }
            m[g] = -INFINITY;
            l[g] = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[g][j] = 0.f;
        }
    }

    __device__ __forceinline__ void consume(uint32_t tk, uint32_t tv, int t0, int u0, int valid,
                                            int rmask, int half_bytes, float scale_log2,
                                            int lane) {
        const int par = lane >> 4, c = lane & 15;
        float s[G][8];
        // ---- logits: each half-warp reduces one token's dot product
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const RowAddr ra = row_addr(tk, t0 + 2 * i + par, rmask);
            const uint4 kv = lds128(chunk_addr(ra, c, half_bytes));
            const uint32_t w[4] = {kv.x, kv.y, kv.z, kv.w};
            float kf[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                kf[2 * j] = bf16_lo(w[j]);
                kf[2 * j + 1] = bf16_hi(w[j]);
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float d = 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) d = fmaf(qf[g][j], kf[j], d);
                d += __shfl_xor_sync(0xffffffffu, d, 1);
                d += __shfl_xor_sync(0xffffffffu, d, 2);
                d += __shfl_xor_sync(0xffffffffu, d, 4);
                d += __shfl_xor_sync(0xffffffffu, d, 8);
                const int tok = u0 + 2 * i + par;
                s[g][i] = tok < valid ? d * scale_log2 : -INFINITY;
            }
        }
        // ---- online softmax (both half-warps share one running max)
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float mx = s[g][0];
#pragma unroll
            for (int i = 1; i < 8; ++i) mx = fmaxf(mx, s[g][i]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mn = fmaxf(m[g], mx);
            const float mu = mn == -INFINITY ? 0.f : mn;
            const float al = fast_exp2(m[g] - mu);
            m[g] = mn;
            float sum = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                s[g][i] = fast_exp2(s[g][i] - mu);
                sum += s[g][i];
            }
            l[g] = l[g] * al + sum;
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[g][j] *= al;
        }
        // ---- accumulate P V over this half-warp's tokens
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int tok = u0 + 2 * i + par;
            if (tok < valid) {
                const RowAddr ra = row_addr(tv, t0 + 2 * i + par, rmask);
                const uint4 vv = lds128(chunk_addr(ra, c, half_bytes));
                const uint32_t w[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
                for (int g = 0; g < G; ++g) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        acc[g][2 * j] = fmaf(s[g][i], bf16_lo(w[j]), acc[g][2 * j]);
                        acc[g][2 * j + 1] = fmaf(s[g][i], bf16_hi(w[j]), acc[g][2 * j + 1]);
                    }
                }
            }
        }
    }

    __device__ __forceinline__ void dump(float* red_m, float* red_l, float* dump, int slice,
                                         int lane) {
        const int par = lane >> 4, c = lane & 15;
        float* base = dump + slice * 16 * kHeadDim;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            // both half-warps used the same running max, so their sums add
            const float lt = l[g] + __shfl_xor_sync(0xffffffffu, l[g], 16);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[g][j] += __shfl_xor_sync(0xffffffffu, acc[g][j], 16);
            if (lane == 0) {
                red_m[slice * 16 + g] = m[g];
                red_l[slice * 16 + g] = lt;
            }
            if (par == 0) {
                float* row = base + g * kHeadDim;
                *reinterpret_cast<float4*>(row + dump_col(g, c * 8)) =
                    make_float4(acc[g][0], acc[g][1], acc[g][2], acc[g][3]);
                *reinterpret_cast<float4*>(row + dump_col(g, c * 8 + 4)) =
                    make_float4(acc[g][4], acc[g][5], acc[g][6], acc[g][7]);
            }
        }
    }
};

// ------------------------------------------------------------------ shared state

template <class C>
struct Smem {
    uint8_t* base;
    __device__ __forceinline__ uint32_t ring(int slot) const {
        return smem_addr(base) + slot * C::kStageBytes;
    }
    __device__ __forceinline__ float* dump(int slot) const {
        return reinterpret_cast<float*>(base + slot * C::kStageBytes);
    }
    __device__ __forceinline__ uint32_t qbuf(int slot) const {
        return smem_addr(base) + C::kQOffset + slot * C::kQBytes;
    }
    __device__ __forceinline__ StageRec* rec(int slot) const {
        return reinterpret_cast<StageRec*>(base + C::kRecOffset) + slot;
    }
    __device__ __forceinline__ uint64_t* full(int slot) const {
        return reinterpret_cast<uint64_t*>(base + C::kBarOffset) + slot;
    }
    __device__ __forceinline__ uint64_t* empty(int slot) const {
        return reinterpret_cast<uint64_t*>(base + C::kBarOffset) + C::kStages + slot;
    }
    // cluster merge: the pieces' states (written remotely into rank 0)
    __device__ __forceinline__ uint32_t cluster_o(int rank, int row) const {
        return smem_addr(base) + C::kClusterOff + (rank * C::kQRows + row) * kHeadDim * 4;
    }
    __device__ __forceinline__ uint32_t cluster_s(int rank, int row) const {
        return smem_addr(base) + C::kClusterOff + C::kClusterOBytes + (rank * C::kQRows + row) * 4;
    }
    // every CTA of the cluster arrives here in rank 0
    __device__ __forceinline__ uint64_t* cluster_bar() const {
        return reinterpret_cast<uint64_t*>(base + C::kBarOffset) + 2 * C::kStages;
    }
    __device__ __forceinline__ int* issued() const {
        return reinterpret_cast<int*>(base + C::kIssuedOffset);
    }
    __device__ __forceinline__ volatile int* flags() const {
        return reinterpret_cast<volatile int*>(base + C::kFlagOffset);
    }
    __device__ __forceinline__ float* red_m() const {
        return reinterpret_cast<float*>(base + C::kRedOffset);
    }
    __device__ __forceinline__ float* red_l() const {
        return red_m() + C::kConsumerWarps * 16;
    }
};

// ------------------------------------------------------------------ the kernel

// Address in cluster rank 0 of the same shared-memory location.
__device__ __forceinline__ uint32_t map_rank0(uint32_t local) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(remote) : "r"(local));
    return remote;
}

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x),
                 "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Rank 0 of a cluster merges row g of the cluster's n pieces from its own
// shared memory (every lane holds all n log2-sums, so no shuffles): the
// state merge of the "Single decode split-K" row, with natural-log weights
// as the merge kernel takes them.
template <class C>
__device__ __forceinline__ void cluster_merge_row(const Smem<C>& sm, int g, int n, int lane,
                                                  uint16_t* out_row, float* lse_out) {
    float sv[kMaxClusterCtas];
    float M = -INFINITY;
#pragma unroll
    for (int i = 0; i < kMaxClusterCtas; ++i) {
        sv[i] = i < n ? lds_f32(sm.cluster_s(i, g)) * kLn2 : -INFINITY;
        M = fmaxf(M, sv[i]);
    }
    float W = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
#pragma unroll
        for (int i = 0; i < kMaxClusterCtas; ++i) {
            if (i < n) {
                const float w = expf(sv[i] - M);
                W += w;
                const uint4 x = lds128(sm.cluster_o(i, g) + lane * 16);
                acc.x = fmaf(w, __uint_as_float(x.x), acc.x);
                acc.y = fmaf(w, __uint_as_float(x.y), acc.y);
                acc.z = fmaf(w, __uint_as_float(x.z), acc.z);
                acc.w = fmaf(w, __uint_as_float(x.w), acc.w);
            }
        }
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    uint2 packed;
    packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(out_row + lane * 4) = packed;
    if (lane == 0 && lse_out != nullptr) *lse_out = W > 0.f ? M + logf(W) : -INFINITY;
}

// kCluster: launched as clusters of p.cluster_c CTAs that merge their
// pieces in rank 0 (a separate instantiation, so the merge code does not
// weigh on the registers of the kernels launched without clusters).
template <class C, class WL, bool kCluster>
__device__ __forceinline__ void decode_body(const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                                            const DecodeParams& p, const WL& work) {
    extern __shared__ uint8_t smem_raw[];
    const Smem<C> sm{reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023))};
    volatile int* flags = sm.flags();  // [0] abort

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ps = p.page_size;
    const int rmask = ps - 1;
    const int half_bytes = ps * 128;
    const int pages_per_stage = C::kStageTokens / ps;
    const int G = p.group;
    // The work list sits in the parameter buffer, unless it was too long or
    // the workspace is bound (then it is in the workspace).
    const int4* units = p.units;
    const int32_t* cta_begin = nullptr;
    if constexpr (std::is_same<WL, WorkList>::value) {
        if (units == nullptr) {
            units = work.unit;
            cta_begin = work.cta_begin;
        }
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(sm.full(s), 1);
            mbar_init(sm.empty(s), C::kConsumerWarps);
            sm.issued()[s] = 0;
        }
        if constexpr (kCluster) mbar_init(sm.cluster_bar(), static_cast<uint32_t>(p.cluster_c));
        flags[0] = 0;
        fence_mbar_init();
    }
    if (warp == C::kConsumerWarps && lane == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
    }
    // Launched as a programmatic dependent of the kernel before it on the
    // stream (a plan with pdl = 1), this CTA may start while that kernel is
    // still running: nothing in global memory is read or written before the
    // wait. Launched plainly, the wait returns at once.
    grid_dependency_wait();
    if (threadIdx.x == 0) {
        if (blockIdx.x == 0) {
            *p.last_epoch = p.epoch;  // whose status the word may hold
            // an unbound run ends any binding of the workspace it writes
            if (p.clear_stamp != nullptr) *p.clear_stamp = 0ull;
        }
        // The kernels behind this one (merge, prefix tiles) may be scheduled
        // now; they wait for this grid before they read its results.
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    }
    __syncthreads();
    // A cluster's barrier in rank 0 is initialised before any CTA can arrive.
    if constexpr (kCluster) cluster_sync_all();

    using Consumer = typename std::conditional<C::kMma, MmaConsumer<C>, FmaConsumer<C>>::type;

    if (warp == C::kConsumerWarps) {
        // ================================================ producer warp
        // This CTA's share of the work is units [u_begin, u_end), in order.
        // The next unit's entry is read after the current unit's first stage
        // is issued and its first page indices after the second, so these
        // dependent loads overlap the current unit's streaming.
        struct Unit {
            int unit;
            int4 it;
            int win, nxt;  // page indices [0, 32) and [32, 64) of the unit, by lane
        };
        // A bound workspace is used only while it still carries this plan's
        // stamp; every unit is bounds-checked before it is used. The CTA's
        // range (and, from a list in memory, its first unit) is read together
        // with the stamp (all lie inside the workspace) and used only if the
        // stamp matches.
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
        int g = 0;  // ring position
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
            const int row0 = ((it.z >> kUnitBBits) & 1) * 16;  // second 16-row half of a group
            const int nrows = min(G - row0, C::kMma ? 16 : G);
            const int hkv = static_cast<int>(static_cast<uint32_t>(it.z) >> (kUnitBBits + 1));
            const int valid = last_len ? (n_pages - 1) * ps + last_len : n_pages * ps;
            int n_stages = (n_pages + pages_per_stage - 1) / pages_per_stage;
            const bool unit_ok = n_pages >= 1 && it.x >= 0 &&
                                 static_cast<int64_t>(it.x) + n_pages <= p.nnz && b < p.batch &&
                                 hkv < p.num_kv_heads && row0 < G && it.w >= -1 &&
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
            if (__any_sync(0xffffffffu, bad) && lane == 0) record_status(p.status, p.epoch, kDeviceBadPage);
            win = bad ? 0 : win;
            for (int s = 0; s < n_stages; ++s, ++g) {
                const int slot = g % C::kStages;
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
                if (lane == 0 && g >= C::kStages)
                    okw = mbar_wait(sm.empty(slot), ((g / C::kStages) + 1) & 1, flags, p.wait_ns)
                              ? 1
                              : 0;
                if (!__shfl_sync(0xffffffffu, okw, 0)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    StageRec* r = sm.rec(slot);
                    r->b = b;
                    r->hkv = hkv;
                    r->valid = valid;
                    r->n_stages = n_stages;
                    r->s = s;
                    r->slot = it.w;
                    r->row0 = row0;
                    r->nrows = nrows;
                    const uint32_t qbytes =
                        s == 0 ? static_cast<uint32_t>(nrows * kHeadDim * 2) : 0u;
                    mbar_arrive_expect_tx(sm.full(slot), npg * ps * kHeadDim * 2 * 2 + qbytes);
                    if (s == 0)
                        bulk_load(sm.qbuf(slot),
                                  p.q + (static_cast<size_t>(b) * p.num_qo_heads + hkv * G +
                                         row0) * kHeadDim,
                                  qbytes, sm.full(slot));
                }
                const uint32_t tk = sm.ring(slot);
                const uint32_t tv = tk + C::kStageBytes / 2;
                const int ca = p.layout == 0 ? hkv : 0;  // coordinates (d, A, B, page):
                const int cb = p.layout == 0 ? 0 : hkv;  // NHD (d, head, token, page)
                {                                        // HND (d, token, head, page)
                    // One copy per (page, tensor, 64-column half), one lane each,
                    // so the whole stage is issued by one warp instruction:
                    // lane 4j + 2t + h copies half h of tensor t (K, V) of page j.
                    const int j = lane >> 2;
                    const int page = __shfl_sync(0xffffffffu, win, (pg0 - win_base + j) & 31);
                    if (lane < 4 * npg) {
                        const uint32_t off = j * ps * 256 + ((lane & 1) ? half_bytes : 0);
                        tma_load_4d(((lane & 2) ? tv : tk) + off, (lane & 2) ? &tmap_v : &tmap_k,
                                    sm.full(slot), (lane & 1) * 64, ca, cb, page);
                    }
                }
                if (lane == 0) sm.issued()[slot] += 1;
                if (s == 0) {
                    load_item(nx);
                    nx_item = true;
                } else if (s == 1) {
                    load_idx(nx);
                    nx_idx = true;
                }
            }
            if (!ok) break;
            if (!nx_item) load_item(nx);
            if (!nx_idx) load_idx(nx);
            if (lane == 0 && unit_ok && ((first_page && ip0 != it.x) ||
                              (last_len && (ip1 != it.x + n_pages || lst != last_len))))
                record_status(p.status, p.epoch, kDevicePlanMismatch);
            cur = nx;
        }
        if (ok) {
            // End marker: a stage whose record says s = -1, completed by a
            // plain arrive (no bytes).
            const int slot = g % C::kStages;
            int okw = 1;
            if (lane == 0) {
                if (g >= C::kStages)
                    okw = mbar_wait(sm.empty(slot), ((g / C::kStages) + 1) & 1, flags, p.wait_ns)
                              ? 1
                              : 0;
                if (okw) {
                    sm.rec(slot)->s = -1;
                    mbar_arrive(sm.full(slot));
                    sm.issued()[slot] += 1;
                }
            }
            ok = __shfl_sync(0xffffffffu, okw, 0) != 0;
        }
        if (!ok && lane == 0) {
            flags[0] = 1;
            record_status(p.status, p.epoch, kDeviceWaitTimeout);
        }
    } else {
        // ================================================ consumer warps
        // Every consumer-only barrier is named barrier 1. The consumer warps
        // always take the same path through it: each stage's wait result is
        // AND-reduced over all of them before anyone acts on it.
        Consumer cs;
        int own_b = -1, own_hkv = 0, own_slot = -1;  // the CTA's unit (cluster merge)
        const int slice = warp % C::kSlices;
        const int mt = warp / C::kSlices;
        const int ctid = threadIdx.x;  // 0 .. kConsumerThreads-1
        bool ok = true;
        for (int g = 0;; ++g) {
            const int slot = g % C::kStages;
            const bool got = mbar_wait(sm.full(slot), (g / C::kStages) & 1, flags, p.wait_ns);
            if (!consumer_all(C::kConsumerThreads, got)) {
                ok = false;
                break;
            }
            const StageRec r = *sm.rec(slot);
            if (r.s < 0) break;
            if (r.s == 0) {
                cs.init(sm.qbuf(slot), r.nrows, mt, lane);
                own_b = r.b;
                own_hkv = r.hkv;
                own_slot = r.slot;
            }
            const int t0 = slice * kSliceTokens;
            const int u0 = r.s * C::kStageTokens + t0;
            if (u0 < r.valid) {
                const uint32_t tk = sm.ring(slot);
                cs.consume(tk, tk + C::kStageBytes / 2, t0, u0, r.valid, rmask, half_bytes,
                           p.scale_log2, lane);
            }
            if (r.s == r.n_stages - 1) {
                // ---- unit epilogue: merge the warps' states through this
                // stage's buffer (held until the end), then write.
                float* dump = sm.dump(slot);
                float* red_m = sm.red_m();
                float* red_l = sm.red_l();
                consumer_sync(C::kConsumerThreads);  // every warp is done reading K/V here
                const int hq0 = r.hkv * G + r.row0;
                for (int round = 0; round < C::kMtiles; ++round) {
                    if (mt == round) cs.dump(red_m, red_l, dump, slice, lane);
                    consumer_sync(C::kConsumerThreads);
                    const int rows = min(16, r.nrows - round * 16);
                    for (int i = ctid; i < rows * (kHeadDim / 4); i += C::kConsumerThreads) {
                        const int rr = i / (kHeadDim / 4);
                        const int d4 = i - rr * (kHeadDim / 4);
                        float M = -INFINITY;
#pragma unroll
                        for (int w = 0; w < C::kSlices; ++w) M = fmaxf(M, red_m[w * 16 + rr]);
                        float L = 0.f;
                        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (M != -INFINITY) {
#pragma unroll
                            for (int w = 0; w < C::kSlices; ++w) {
                                const float sc = fast_exp2(red_m[w * 16 + rr] - M);
                                L += red_l[w * 16 + rr] * sc;
                                const float4 a = *reinterpret_cast<const float4*>(
                                    dump + (w * 16 + rr) * kHeadDim + dump_col(rr, d4 * 4));
                                o.x += a.x * sc;
                                o.y += a.y * sc;
                                o.z += a.z * sc;
                                o.w += a.w * sc;
                            }
                        }
                        float lse2 = -INFINITY;
                        if (L > 0.f) {
                            const float inv = 1.f / L;
                            o.x *= inv;
                            o.y *= inv;
                            o.z *= inv;
                            o.w *= inv;
                            lse2 = M + __log2f(L);
                        }
                        const int hq = hq0 + round * 16 + rr;
                        if (r.slot < 0) {
                            const size_t row = static_cast<size_t>(r.b) * p.num_qo_heads + hq;
                            uint2 packed;
                            packed.x = pack_bf16x2(o.x, o.y);
                            packed.y = pack_bf16x2(o.z, o.w);
                            *reinterpret_cast<uint2*>(p.out + row * kHeadDim + d4 * 4) = packed;
                            if (d4 == 0 && p.lse != nullptr) p.lse[row] = lse2 * kLn2;
                        } else if constexpr (kCluster) {
                            // this piece's state, into rank 0's shared memory
                            const uint32_t rank = cluster_ctarank();
                            st_cluster_v4(map_rank0(sm.cluster_o(static_cast<int>(rank), rr) +
                                                    d4 * 16),
                                          o);
                            if (d4 == 0)
                                st_cluster_f32(map_rank0(sm.cluster_s(static_cast<int>(rank), rr)),
                                               lse2);
                        } else {
                            // partial states are [slot][G][128]
                            const size_t row =
                                static_cast<size_t>(r.slot) * G + r.row0 + round * 16 + rr;
                            *reinterpret_cast<float4*>(p.part_o + row * kHeadDim + d4 * 4) = o;
                            if (d4 == 0) p.part_lse[row] = lse2;
                        }
                    }
                    consumer_sync(C::kConsumerThreads);  // dump reads done before reuse
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.empty(slot));
        }
        if (!ok && lane == 0) {
            flags[0] = 1;
            record_status(p.status, p.epoch, kDeviceWaitTimeout);
        }
        if constexpr (kCluster) {
            // ---- cluster merge: this CTA's piece (its partial state is
            // written: every consumer passed the epilogue's last barrier) is
            // announced to rank 0, which merges the cluster's pieces.
            consumer_sync(C::kConsumerThreads);
            if (ctid == 0) mbar_arrive_remote(sm.cluster_bar(), 0);
            if (cluster_ctarank() == 0) {
                const bool got = mbar_wait_cluster(sm.cluster_bar(), 0, 4 * p.wait_ns);
                if (consumer_all(C::kConsumerThreads, got)) {
                    if (own_b >= 0) {
                        const size_t row0 =
                            static_cast<size_t>(own_b) * p.num_qo_heads + own_hkv * G;
                        for (int g = warp; g < G; g += C::kConsumerWarps)
                            cluster_merge_row(sm, g, p.cluster_c, lane,
                                              p.out + (row0 + g) * kHeadDim,
                                              p.lse != nullptr ? p.lse + row0 + g : nullptr);
                    }
                } else if (ctid == 0) {
                    record_status(p.status, p.epoch, kDeviceWaitTimeout);
                }
            }
        }
    }
    __syncthreads();  // every warp has left its loop
    // No CTA of a cluster leaves before all have passed this point: a piece
    // stores into rank 0's shared memory and arrives there before it gets
    // here, and its arrival releases those operations, so rank 0 (even one
    // whose wait for the pieces gave up) never exits ahead of a remote store.
    // Rank 0 orders nothing of its own by this barrier: its arrival is
    // relaxed (a release there would wait for its output stores, +1.5 us on a
    // one-request batch). Every wait before it is bounded, so it completes.
    if constexpr (kCluster) {
        if (cluster_ctarank() == 0)
            cluster_sync_relaxed_arrive();
        else
            cluster_sync_all();
    }

    if (flags[0] && threadIdx.x == 0) {
        // Aborted: wait (bounded) for the copies already issued, then leave.
        for (int s = 0; s < C::kStages; ++s)
            if (sm.issued()[s] > 0)
                mbar_wait(sm.full(s), (sm.issued()[s] - 1) & 1, nullptr, kWaitTimeoutNs);
    }
}

// The decode kernel, in its two register budgets (Cfg::kRegs168).
template <class C, class WL, bool kCluster>
__global__ void __launch_bounds__(C::kThreads)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_v,
                        const __grid_constant__ DecodeParams p,
                        const __grid_constant__ WL work) {
    decode_body<C, WL, kCluster>(tmap_k, tmap_v, p, work);
}

template <class C, class WL, bool kCluster>
__global__ void __maxnreg__(168)
    paged_decode_kernel_r168(const __grid_constant__ CUtensorMap tmap_k,
                             const __grid_constant__ CUtensorMap tmap_v,
                             const __grid_constant__ DecodeParams p,
                             const __grid_constant__ WL work) {
    decode_body<C, WL, kCluster>(tmap_k, tmap_v, p, work);
}

template <class C, class WL>
using KernelFn = void (*)(const CUtensorMap, const CUtensorMap, const DecodeParams, const WL);

template <class C, class WL, bool kCluster = false>
KernelFn<C, WL> kernel_of() {
    if constexpr (C::kRegs168) return paged_decode_kernel_r168<C, WL, kCluster>;
    else return paged_decode_kernel<C, WL, kCluster>;
}

// cudaFuncSetAttribute is per device; remember which devices are set up.
template <class C, class WL, bool kCluster = false>
cudaError_t ensure_smem_attribute() {
    static std::atomic<uint64_t> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit != 0 && (done.load(std::memory_order_relaxed) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel_of<C, WL, kCluster>(),
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kCluster ? C::kSmemBytesCluster : C::kSmemBytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_relaxed);
    return e;
}

template <class C, class WL, bool cluster>
cudaError_t launch_ex(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                      const WL& w, int grid, cudaStream_t stream, bool pdl) {
    cudaError_t e = ensure_smem_attribute<C, WL, cluster>();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = cluster ? C::kSmemBytesCluster : C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if constexpr (cluster) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = static_cast<unsigned>(p.cluster_c);
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl) {
        // a programmatic dependent of the kernel before it on the stream: it
        // may start early and waits (griddepcontrol.wait) before touching memory
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel_of<C, WL, cluster>(), tk, tv, p, w);
}

template <class C>
cudaError_t launch(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                   const WorkList* w, int grid, cudaStream_t stream, bool pdl) {
    if (p.cluster_c > 1) {
        // clusters of p.cluster_c CTAs (CUDA-core and 8-row variants); grid is a
        // multiple of it
        if constexpr (C::kMma && C::kHiRows) {
            return cudaErrorInvalidValue;  // 16-row groups: no cluster merge
        } else {
            using CC = typename ClusterCfg<C>::type;
            static_assert(CC::kSmemBytesCluster <= 113 * 1024, "two cluster CTAs a SM");
            if (grid % p.cluster_c != 0 || p.cluster_c > kMaxClusterCtas)
                return cudaErrorInvalidValue;
            if (w != nullptr)
                return launch_ex<CC, WorkList, true>(tk, tv, p, *w, grid, stream, pdl);
            return launch_ex<CC, NoList, true>(tk, tv, p, NoList{0}, grid, stream, pdl);
        }
    }
    if (w != nullptr) return launch_ex<C, WorkList, false>(tk, tv, p, *w, grid, stream, pdl);
    return launch_ex<C, NoList, false>(tk, tv, p, NoList{0}, grid, stream, pdl);
}

template <class C>
VariantShape shape_of() {
    return {C::kThreads, C::kStageTokens, C::kStages, C::kSmemBytes};
}

template <class C>
cudaError_t occupancy_of(int* n) {
    cudaError_t e = ensure_smem_attribute<C, WorkList>();
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, kernel_of<C, WorkList>(),
                                                         C::kThreads, C::kSmemBytes);
}

}  // namespace

VariantShape variant_shape(int variant) {
    switch (variant) {
        case kVariantFmaG1: return shape_of<CfgFmaG1>();
        case kVariantFmaG2: return shape_of<CfgFmaG2>();
        case kVariantMma8: return shape_of<CfgMma8>();
        case kVariantMma16: return shape_of<CfgMma16>();
        case kVariantWide: return wide_shape();
        default: return shape_of<CfgMma16>();  // kVariantMma32: two 16-row CTAs per piece
    }
}

cudaError_t variant_occupancy(int variant, int* n) {
    switch (variant) {
        case kVariantFmaG1: return occupancy_of<CfgFmaG1>(n);
        case kVariantFmaG2: return occupancy_of<CfgFmaG2>(n);
        case kVariantMma8: return occupancy_of<CfgMma8>(n);
        case kVariantMma16: return occupancy_of<CfgMma16>(n);
        case kVariantWide: return wide_occupancy(n);
        default: return occupancy_of<CfgMma16>(n);
    }
}

cudaError_t launch_decode(int variant, const CUtensorMap& tk, const CUtensorMap& tv,
                          const DecodeParams& p, const WorkList* w, int grid,
                          cudaStream_t stream, bool pdl) {
    switch (variant) {
        case kVariantFmaG1: return launch<CfgFmaG1>(tk, tv, p, w, grid, stream, pdl);
        case kVariantFmaG2: return launch<CfgFmaG2>(tk, tv, p, w, grid, stream, pdl);
        case kVariantMma8: return launch<CfgMma8>(tk, tv, p, w, grid, stream, pdl);
        case kVariantMma16: return launch<CfgMma16>(tk, tv, p, w, grid, stream, pdl);
        default: return launch<CfgMma16>(tk, tv, p, w, grid, stream, pdl);
    }
}

}  // namespace oxd
