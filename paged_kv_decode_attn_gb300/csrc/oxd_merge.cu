// Attention-state merge for sm_103a ("FlashInfer parity matrix" page,
// "Domain coverage": attention state and cascade, state merge; and the merge
// step of the "Single decode split-K" row of "Admitted attention matrix").
//
// For one output row it combines states (v_i, s_i):
//   M = max_i s_i, w_i = exp(s_i - M), v = sum w_i v_i / sum w_i,
//   s = M + ln sum w_i,
// with -inf states weighing nothing and an all -inf row giving v = 0,
// s = -inf. One warp per output row; each lane owns 4 consecutive columns
// (16-byte loads); the states are visited in order, so the result is
// deterministic. The same kernel serves oxd_merge_states (uniform state
// counts) and the decode run's split streams (an entry list; launched behind
// the decode kernel, it first waits for that grid to complete).
#include <cuda_bf16.h>

#include <type_traits>

#include "oxd_internal.h"

namespace oxd {
namespace {

constexpr int kWarpsPerBlock = 4;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void merge_row(const MergeParams& p, const int4* entries) {
    const int lane = threadIdx.x & 31;
    const long long gw = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
    if (gw >= static_cast<long long>(p.n) * p.R) return;
    const int n = static_cast<int>(gw / p.R);
    const int r = static_cast<int>(gw - static_cast<long long>(n) * p.R);
    long long row0 = static_cast<long long>(n) * p.R;
    long long first = static_cast<long long>(n) * p.S;
    int count = p.S;
    if (!p.uniform) {
        const int4 e = entries[n];
        row0 = e.x;
        first = e.y;
        count = e.z;
        // entries of a bound workspace are checked before use
        if (row0 < 0 || row0 + p.R > p.n_rows || first < 0 || count < 0 ||
            (first + count) * p.R > p.n_states)
            return;
    }
    const float* s = p.s + first * p.R + r;     // state i at s[i * R]
    const float* v = p.v + (first * p.R + r) * p.D;  // state i at v[i * R * D]
    // pass 1: maximum LSE over the states (lanes stride over them)
    float M = -INFINITY;
    for (int i = lane; i < count; i += 32) M = fmaxf(M, s[static_cast<size_t>(i) * p.R] * p.s_to_ln);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float W = 0.f;
    if (M != -INFINITY) {
        for (int i = lane; i < count; i += 32)
            W += expf(s[static_cast<size_t>(i) * p.R] * p.s_to_ln - M);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    const size_t vstride = static_cast<size_t>(p.R) * p.D;
    // pass 2: weighted sum, states in order
    for (int c = lane * 4; c < p.D; c += 128) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) {
#pragma unroll 4
            for (int i = 0; i < count; ++i) {
                const float w = expf(s[static_cast<size_t>(i) * p.R] * p.s_to_ln - M);
                const float4 x = *reinterpret_cast<const float4*>(v + i * vstride + c);
                acc.x = fmaf(w, x.x, acc.x);
                acc.y = fmaf(w, x.y, acc.y);
                acc.z = fmaf(w, x.z, acc.z);
                acc.w = fmaf(w, x.w, acc.w);
            }
        }
        uint2 packed;
        packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
        packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2*>(p.out + static_cast<size_t>(row0 + r) * p.D + c) = packed;
    }
    if (lane == 0 && p.lse != nullptr)
        p.lse[row0 + r] = W > 0.f ? M + logf(W) : -INFINITY;
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32) merge_kernel(const MergeParams p) {
    merge_row(p, nullptr);
}

template <class SL>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    split_merge_kernel(const MergeParams p, const __grid_constant__ SL inl) {
    // Behind the decode kernel this waits for its grid to complete and its
    // writes to be visible; launched on its own it returns at once.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (p.ws_stamp != nullptr && *p.ws_stamp != p.stamp) return;  // not this plan's entries
    const int4* entries = p.entries;
    if constexpr (std::is_same<SL, SplitList>::value) {
        if (entries == nullptr) entries = inl.entry;
    }
    merge_row(p, entries);
}

unsigned blocks_for(const MergeParams& p) {
    const long long warps = static_cast<long long>(p.n) * p.R;
    const long long blocks = (warps + kWarpsPerBlock - 1) / kWarpsPerBlock;
    return blocks > 0x7fffffffLL ? 0u : static_cast<unsigned>(blocks);
}

}  // namespace

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream) {
    const unsigned blocks = blocks_for(p);
    if (blocks == 0) return cudaErrorInvalidConfiguration;
    merge_kernel<<<blocks, kWarpsPerBlock * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_split_merge(const MergeParams& p, const SplitList* splits,
                               cudaStream_t stream, bool early) {
    const unsigned blocks = blocks_for(p);
    if (blocks == 0) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(kWarpsPerBlock * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = early ? 1 : 0;
    if (splits != nullptr) return cudaLaunchKernelEx(&cfg, split_merge_kernel<SplitList>, p, *splits);
    return cudaLaunchKernelEx(&cfg, split_merge_kernel<NoList>, p, NoList{0});
}

}  // namespace oxd
