// Attention-state merge for sm_103a ("FlashInfer parity matrix" page,
// "Domain coverage": attention state and cascade, state merge; and the merge
// step of the "Single decode split-K" row of "Admitted attention matrix").
//
// One warp per output row merges its states with merge_states_row
// (oxd_merge_row.cuh). The same kernel serves oxd_merge_states (uniform state
// counts) and the decode run's split streams with more pieces than the
// decode kernel merges itself (an entry list; launched behind the decode
// kernel, it first waits for that grid to complete).
#include <cuda_bf16.h>

#include <type_traits>

#include "oxd_internal.h"
#include "oxd_merge_row.cuh"

namespace oxd {
namespace {

constexpr int kWarpsPerBlock = 4;

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
    // state i of row r: s[(first + i) * R + r], v[((first + i) * R + r) * D]
    merge_states_row(p.s + first * p.R + r, static_cast<size_t>(p.R),
                     p.v + (first * p.R + r) * p.D, static_cast<size_t>(p.R) * p.D, count, p.D,
                     p.s_to_ln, p.out + static_cast<size_t>(row0 + r) * p.D,
                     p.lse != nullptr ? p.lse + row0 + r : nullptr, lane);
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
