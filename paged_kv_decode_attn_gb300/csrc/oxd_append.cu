// Fused rotary embedding + paged KV append for sm_103a ("FlashInfer parity
// matrix" page, "Admitted attention matrix", rows "Standard RoPE" (D128 NeoX
// split-half with explicit int32 positions) and "Fused RoPE plus paged
// append"; "Paged KV ownership difference": the append writes only pages
// whose reference count is one).
//
// One warp per row: a query head of a token (RoPE into q_out) or a KV head
// of a token (RoPE of K, copy of V, into the token's page slot). Lane l owns
// the pairs (2l, 64 + 2l) and (2l + 1, 64 + 2l + 1): two 4-byte loads and
// stores of 32 contiguous lanes each per half row. The rotation angle is
// formed in double (position times a frequency computed on the host in
// double), its cosine and sine rounded to float, the products done in float
// and the result rounded once to bf16. A KV row whose request or position
// lies outside the block table, whose page index lies outside the pool, or
// whose page is shared (reference count not one) is not written; the run's
// status word records why.
#include <cuda_bf16.h>

#include "oxd_internal.h"
#include "oxd_ptx.cuh"

namespace oxd {
namespace {

constexpr int kAppendWarps = 4;
constexpr int kDeviceSharedPage = 4;
constexpr int kDeviceBadPosition = 5;

__device__ __forceinline__ void rope_pairs(const uint16_t* src, uint16_t* dst, int pos,
                                           const double* freq, int lane) {
    const uint32_t lo = *reinterpret_cast<const uint32_t*>(src + 2 * lane);
    const uint32_t hi = *reinterpret_cast<const uint32_t*>(src + 64 + 2 * lane);
    float x[2] = {__uint_as_float(lo << 16), __uint_as_float(lo & 0xffff0000u)};
    float y[2] = {__uint_as_float(hi << 16), __uint_as_float(hi & 0xffff0000u)};
    float a[2], b[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        double s, c;
        sincos(static_cast<double>(pos) * freq[2 * lane + j], &s, &c);
        const float cf = static_cast<float>(c), sf = static_cast<float>(s);
        a[j] = x[j] * cf - y[j] * sf;  // first half
        b[j] = y[j] * cf + x[j] * sf;  // second half
    }
    __nv_bfloat162 ra = __floats2bfloat162_rn(a[0], a[1]);
    __nv_bfloat162 rb = __floats2bfloat162_rn(b[0], b[1]);
    *reinterpret_cast<uint32_t*>(dst + 2 * lane) = *reinterpret_cast<uint32_t*>(&ra);
    *reinterpret_cast<uint32_t*>(dst + 64 + 2 * lane) = *reinterpret_cast<uint32_t*>(&rb);
}

__global__ void __launch_bounds__(kAppendWarps * 32) rope_append_kernel(const AppendParams p) {
    if (blockIdx.x == 0 && threadIdx.x == 0) *p.last_epoch = p.epoch;
    const int lane = threadIdx.x & 31;
    const long long row = static_cast<long long>(blockIdx.x) * kAppendWarps + (threadIdx.x >> 5);
    const long long q_rows = static_cast<long long>(p.T) * p.Hq;
    if (row < q_rows) {
        const int t = static_cast<int>(row / p.Hq);
        const size_t off = static_cast<size_t>(row) * kHeadDim;
        rope_pairs(p.q + off, p.q_out + off, p.positions[t], p.freq, lane);
        return;
    }
    const long long kv = row - q_rows;
    if (kv >= static_cast<long long>(p.T) * p.Hkv) return;
    const int t = static_cast<int>(kv / p.Hkv);
    const int h = static_cast<int>(kv - static_cast<long long>(t) * p.Hkv);
    const int b = p.token_request[t];
    const int pos = p.positions[t];
    int code = 0;
    int64_t page = -1;
    int lo = 0, hi = 0;
    if (b >= 0 && b < p.B) {
        lo = p.indptr[b];
        hi = p.indptr[b + 1];
    }
    if (b < 0 || b >= p.B || lo < 0 || hi < lo || hi > p.num_indices || pos < 0 ||
        static_cast<int64_t>(pos) >= static_cast<int64_t>(hi - lo) * p.page_size) {
        code = kDeviceBadPosition;
    } else {
        page = p.indices[lo + pos / p.page_size];
        if (page < 0 || page >= p.num_pages)
            code = kDeviceBadPage;
        else if (p.refcount[page] != 1)
            code = kDeviceSharedPage;
    }
    if (code != 0) {
        if (lane == 0) record_status(p.status, p.epoch, code);
        return;
    }
    const int slot = pos % p.page_size;
    const size_t dst =
        (p.layout == 0
             ? (static_cast<size_t>(page) * p.page_size + slot) * p.Hkv + h
             : (static_cast<size_t>(page) * p.Hkv + h) * p.page_size + slot) *
        kHeadDim;
    const size_t src = static_cast<size_t>(kv) * kHeadDim;
    rope_pairs(p.k + src, p.k_pages + dst, pos, p.freq, lane);
    // V unchanged: 256 bytes, 8 per lane
    *reinterpret_cast<uint2*>(p.v_pages + dst + 4 * lane) =
        *reinterpret_cast<const uint2*>(p.v + src + 4 * lane);
}

}  // namespace

cudaError_t launch_rope_append(const AppendParams& p, cudaStream_t stream) {
    const long long rows = static_cast<long long>(p.T) * (p.Hq + p.Hkv);
    const long long blocks = (rows + kAppendWarps - 1) / kAppendWarps;
    if (blocks < 1 || blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    rope_append_kernel<<<static_cast<unsigned>(blocks), kAppendWarps * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace oxd
