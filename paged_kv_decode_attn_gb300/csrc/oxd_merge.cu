// Attention-state merge for sm_103a ("FlashInfer parity matrix" page,
// "Domain coverage": attention state and cascade, state merge). The decode
// kernel merges its own split partitions in place; this kernel serves the
// public oxd_merge_states entry point.
//
// For one row (request) and head h it combines S states (v_i, s_i):
//   M = max_i s_i, w_i = exp(s_i - M), v = sum w_i v_i / sum w_i,
//   s = M + ln sum w_i,
// with -inf states weighing nothing and an all -inf row giving v = 0,
// s = -inf. One warp per (row, head); each lane owns 4 consecutive columns
// (16-byte loads); the states are visited in order, so the result is
// deterministic.
#include <cuda_bf16.h>

#include "oxd_internal.h"

namespace oxd {
namespace {

constexpr int kWarpsPerBlock = 4;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void merge_rows(const MergeParams& p, const int4* split);

__global__ void __launch_bounds__(kWarpsPerBlock * 32) merge_kernel(const MergeParams p) {
    merge_rows(p, nullptr);
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    split_merge_kernel(const MergeParams p, const __grid_constant__ InlineSplits inl) {
    // Behind the decode kernel this waits for its grid to complete and its
    // writes to be visible; launched on its own it returns at once.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    merge_rows(p, p.split != nullptr ? p.split : inl.split);
}

__device__ __forceinline__ void merge_rows(const MergeParams& p, const int4* split) {
    const int lane = threadIdx.x & 31;
    const long long gw = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
    if (gw >= static_cast<long long>(p.n) * p.H) return;
    const int n = static_cast<int>(gw / p.H);
    const int h = static_cast<int>(gw - static_cast<long long>(n) * p.H);
    int row = n, first = n * p.S, count = p.S;
    if (split != nullptr) {
        const int4 sr = split[n];
        row = sr.x;
        first = sr.y;
        count = sr.z;
    }
    // pass 1: maximum LSE over the states (lanes stride over them)
    float M = -INFINITY;
    for (int i = lane; i < count; i += 32)
        M = fmaxf(M, p.s[static_cast<size_t>(first + i) * p.H + h] * p.s_to_ln);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float W = 0.f;
    if (M != -INFINITY) {
        for (int i = lane; i < count; i += 32)
            W += expf(p.s[static_cast<size_t>(first + i) * p.H + h] * p.s_to_ln - M);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    // pass 2: weighted sum, states in order
    for (int c = lane * 4; c < p.D; c += 128) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) {
            for (int i = 0; i < count; ++i) {
                const size_t st = static_cast<size_t>(first + i) * p.H + h;
                const float w = expf(p.s[st] * p.s_to_ln - M);
                const float4 v = *reinterpret_cast<const float4*>(p.v + st * p.D + c);
                acc.x = fmaf(w, v.x, acc.x);
                acc.y = fmaf(w, v.y, acc.y);
                acc.z = fmaf(w, v.z, acc.z);
                acc.w = fmaf(w, v.w, acc.w);
            }
        }
        uint2 packed;
        packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
        packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2*>(p.out + (static_cast<size_t>(row) * p.H + h) * p.D + c) = packed;
    }
    if (lane == 0 && p.lse != nullptr)
        p.lse[static_cast<size_t>(row) * p.H + h] = W > 0.f ? M + logf(W) : -INFINITY;
}

}  // namespace

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream) {
    const long long warps = static_cast<long long>(p.n) * p.H;
    const long long blocks = (warps + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    merge_kernel<<<static_cast<unsigned>(blocks), kWarpsPerBlock * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_split_merge(const MergeParams& p, const InlineSplits& splits,
                               cudaStream_t stream, bool early) {
    const long long warps = static_cast<long long>(p.n) * p.H;
    const long long blocks = (warps + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(kWarpsPerBlock * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = early ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, split_merge_kernel, p, splits);
}

}  // namespace oxd
