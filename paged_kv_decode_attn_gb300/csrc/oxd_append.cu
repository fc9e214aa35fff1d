// Fused rotary embedding + paged KV append for sm_103a ("FlashInfer parity
// matrix" page, "Admitted attention matrix", rows "Standard RoPE" (D128 NeoX
// split-half with explicit int32 positions) and "Fused RoPE plus paged
// append"; "Paged KV ownership difference": the append writes only pages
// whose reference count is one).
//
// A warp takes up to eight heads of one token: either KV heads (RoPE of K,
// copy of V, into the token's page slot, behind the block-table walk) or
// query heads (RoPE into q_out, no table access). Lane l owns the
// pairs (2l, 64 + 2l) and (2l + 1, 64 + 2l + 1): two 4-byte loads and stores
// of 32 contiguous lanes each per half row. The rotation angle is
// kept in turns, pos * f / (2 pi), as a two-float product: the frequency in
// turns comes from the host as hi + lo floats of its double value, the
// rounding error of pos * hi is recovered exactly with an FMA, and the
// nearest whole turn is removed before sincospif, so the angle is accurate to
// about 1e-8 turns for every position below 2^24 without double arithmetic.
// The rotation itself is done in float and rounded once to bf16. A KV row
// whose request or position lies outside the block table, whose page index
// lies outside the pool, or whose page is shared (reference count not one) is
// not written; the run's status word records why.
#include <cuda_bf16.h>

#include "oxd_internal.h"
#include "oxd_ptx.cuh"

namespace oxd {
namespace {

constexpr int kAppendWarps = 8;
constexpr int kKvRows = 8;  // K/V rows (KV heads of one token) per KV warp
constexpr int kQRows = 8;   // query rows (heads of one token) per query warp
constexpr int kDeviceSharedPage = 4;
constexpr int kDeviceBadPosition = 5;

// cos and sin of the angles of this lane's two pairs (2l, 2l + 1) at `pos`.
__device__ __forceinline__ void rope_angles(int pos, const float* turns_hi, const float* turns_lo,
                                            int lane, float (&c)[2], float (&s)[2]) {
    const float P = static_cast<float>(pos);  // exact below 2^24
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const float gh = turns_hi[2 * lane + j], gl = turns_lo[2 * lane + j];
        const float th = P * gh;
        const float tl = fmaf(P, gl, fmaf(P, gh, -th));  // P*gl + rounding error of P*gh
        const float r = (th - rintf(th)) + tl;           // turns, within [-0.5, 0.5]
        sincospif(2.f * r, &s[j], &c[j]);
    }
}

// Rotates the two pairs a lane holds of one 128-wide row (elements 2l, 2l+1
// in `lo`, 64+2l, 64+2l+1 in `hi`) and stores them.
__device__ __forceinline__ void rope_store(uint32_t lo, uint32_t hi, uint16_t* dst,
                                           const float (&c)[2], const float (&s)[2], int lane) {
    const float x0 = __uint_as_float(lo << 16), x1 = __uint_as_float(lo & 0xffff0000u);
    const float y0 = __uint_as_float(hi << 16), y1 = __uint_as_float(hi & 0xffff0000u);
    __nv_bfloat162 ra = __floats2bfloat162_rn(x0 * c[0] - y0 * s[0], x1 * c[1] - y1 * s[1]);
    __nv_bfloat162 rb = __floats2bfloat162_rn(y0 * c[0] + x0 * s[0], y1 * c[1] + x1 * s[1]);
    *reinterpret_cast<uint32_t*>(dst + 2 * lane) = *reinterpret_cast<uint32_t*>(&ra);
    *reinterpret_cast<uint32_t*>(dst + 64 + 2 * lane) = *reinterpret_cast<uint32_t*>(&rb);
}

// Warps of two kinds share one grid. KV warps come first (their work waits
// on the block-table walk, request -> indptr -> page index -> reference
// count, three dependent loads): KV warp (t, c) loads the K and V rows of
// heads [c * kKvRows, ...) of token t, walks the table while they are in
// flight, and stores the rotated K and the V rows in the token's page slot.
// Query warps never touch the table: query warp (t, c) loads the rows of
// heads [c * kQRows, ...) of token t, rotates them and stores them into
// q_out. Each warp loads all its rows before its first store (q_out may be q
// itself, so the compiler could not hoist a later load over an earlier
// store) and forms the token's angles once.
__global__ void __launch_bounds__(kAppendWarps * 32) rope_append_kernel(const AppendParams p) {
    // A decode launched behind this kernel as its programmatic dependent may
    // be scheduled now; it waits for this grid to complete before it touches
    // memory, so it still reads the rotated q and the appended rows.
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (blockIdx.x == 0 && threadIdx.x == 0) *p.last_epoch = p.epoch;
    const int lane = threadIdx.x & 31;
    const long long gw = static_cast<long long>(blockIdx.x) * kAppendWarps + (threadIdx.x >> 5);
    const int kv_chunks = (p.Hkv + kKvRows - 1) / kKvRows;
    const int q_chunks = (p.Hq + kQRows - 1) / kQRows;
    const long long n_kv = static_cast<long long>(p.T) * kv_chunks;
    float c[2], s[2];
    if (gw < n_kv) {
        const int t = static_cast<int>(gw / kv_chunks);
        const int h0 = static_cast<int>(gw - static_cast<long long>(t) * kv_chunks) * kKvRows;
        const int nh = min(kKvRows, p.Hkv - h0);
        const int pos = p.positions[t];
        const int b = p.token_request[t];
        const size_t kv0 = (static_cast<size_t>(t) * p.Hkv + h0) * kHeadDim;
        uint32_t lo[kKvRows], hi[kKvRows];
        uint2 vv[kKvRows];
#pragma unroll
        for (int i = 0; i < kKvRows; ++i) {
            if (i < nh) {
                const uint16_t* src = p.k + kv0 + static_cast<size_t>(i) * kHeadDim;
                lo[i] = *reinterpret_cast<const uint32_t*>(src + 2 * lane);
                hi[i] = *reinterpret_cast<const uint32_t*>(src + 64 + 2 * lane);
                vv[i] = *reinterpret_cast<const uint2*>(p.v + kv0 + static_cast<size_t>(i) * kHeadDim +
                                                        4 * lane);
            }
        }
        int code = 0;
        int64_t page = -1;
        int lo_i = 0, hi_i = 0;
        if (b >= 0 && b < p.B) {
            lo_i = p.indptr[b];
            hi_i = p.indptr[b + 1];
        }
        if (b < 0 || b >= p.B || lo_i < 0 || hi_i < lo_i || hi_i > p.num_indices || pos < 0 ||
            pos >= (1 << 24) ||
            static_cast<int64_t>(pos) >= static_cast<int64_t>(hi_i - lo_i) * p.page_size) {
            code = kDeviceBadPosition;
        } else {
            page = p.indices[lo_i + pos / p.page_size];
            if (page < 0 || page >= p.num_pages)
                code = kDeviceBadPage;
            else if (p.refcount[page] != 1)
                code = kDeviceSharedPage;
        }
        if (code != 0) {
            if (h0 == 0 && lane == 0) record_status(p.status, p.epoch, code);
            return;
        }
        const int slot = pos % p.page_size;
        rope_angles(pos, p.turns_hi, p.turns_lo, lane, c, s);
#pragma unroll
        for (int i = 0; i < kKvRows; ++i) {
            if (i < nh) {
                const int h = h0 + i;
                const size_t dst =
                    (p.layout == 0
                         ? (static_cast<size_t>(page) * p.page_size + slot) * p.Hkv + h
                         : (static_cast<size_t>(page) * p.Hkv + h) * p.page_size + slot) *
                    kHeadDim;
                rope_store(lo[i], hi[i], p.k_pages + dst, c, s, lane);
                *reinterpret_cast<uint2*>(p.v_pages + dst + 4 * lane) = vv[i];
            }
        }
        return;
    }
    const long long g = gw - n_kv;
    if (g >= static_cast<long long>(p.T) * q_chunks) return;
    const int t = static_cast<int>(g / q_chunks);
    const int h0 = static_cast<int>(g - static_cast<long long>(t) * q_chunks) * kQRows;
    const int nh = min(kQRows, p.Hq - h0);
    const int pos = p.positions[t];
    const size_t q0 = (static_cast<size_t>(t) * p.Hq + h0) * kHeadDim;
    uint32_t lo[kQRows], hi[kQRows];
#pragma unroll
    for (int i = 0; i < kQRows; ++i) {
        if (i < nh) {
            const uint16_t* src = p.q + q0 + static_cast<size_t>(i) * kHeadDim;
            lo[i] = *reinterpret_cast<const uint32_t*>(src + 2 * lane);
            hi[i] = *reinterpret_cast<const uint32_t*>(src + 64 + 2 * lane);
        }
    }
    // a position outside [0, 2^24) is refused by the KV warps; its query
    // rows are rotated at the low 24 bits
    rope_angles(pos & ((1 << 24) - 1), p.turns_hi, p.turns_lo, lane, c, s);
#pragma unroll
    for (int i = 0; i < kQRows; ++i)
        if (i < nh) rope_store(lo[i], hi[i], p.q_out + q0 + static_cast<size_t>(i) * kHeadDim, c, s, lane);
}

}  // namespace

cudaError_t launch_rope_append(const AppendParams& p, cudaStream_t stream) {
    if (p.T < 1 || p.Hq < 1 || p.Hkv < 1) return cudaErrorInvalidConfiguration;
    const long long warps = static_cast<long long>(p.T) * ((p.Hkv + kKvRows - 1) / kKvRows) +
                            static_cast<long long>(p.T) * ((p.Hq + kQRows - 1) / kQRows);
    const long long blocks = (warps + kAppendWarps - 1) / kAppendWarps;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    rope_append_kernel<<<static_cast<unsigned>(blocks), kAppendWarps * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace oxd
