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

// The output row this warp merges: its first output row, first state and
// state count; false when the warp has none (or its entry is out of range).
struct RowJob {
    long long row0, first;
    int r, count;
};

__device__ __forceinline__ bool locate_row(const MergeParams& p, const int4* entries, RowJob* j) {
    const long long gw = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
    if (gw >= static_cast<long long>(p.n) * p.R) return false;
    const int n = static_cast<int>(gw / p.R);
    j->r = static_cast<int>(gw - static_cast<long long>(n) * p.R);
    j->row0 = static_cast<long long>(n) * p.R;
    j->first = static_cast<long long>(n) * p.S;
    j->count = p.S;
    if (!p.uniform) {
        const int4 e = entries[n];
        j->row0 = e.x;
        j->first = e.y;
        j->count = e.z;
        // entries of a bound workspace are checked before use
        if (e.x < 0 || j->row0 + p.R > p.n_rows || e.y < 0 || e.z < 0 ||
            (j->first + e.z) * p.R > p.n_states)
            return false;
    }
    return true;
}

__device__ __forceinline__ void merge_row(const MergeParams& p, const RowJob& j) {
    // state i of row r: s[(first + i) * R + r], v[((first + i) * R + r) * D]
    merge_states_row(p.s + j.first * p.R + j.r, static_cast<size_t>(p.R),
                     p.v + (j.first * p.R + j.r) * p.D, static_cast<size_t>(p.R) * p.D, j.count,
                     p.D, p.s_to_ln, p.out + static_cast<size_t>(j.row0 + j.r) * p.D,
                     p.lse != nullptr ? p.lse + j.row0 + j.r : nullptr, threadIdx.x & 31);
}

__global__ void __launch_bounds__(kWarpsPerBlock * 32) merge_kernel(const MergeParams p) {
    RowJob j;
    if (locate_row(p, nullptr, &j)) merge_row(p, j);
}

template <class SL>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    split_merge_kernel(const MergeParams p, const __grid_constant__ SL inl) {
    // The entry list and the stamp were written before the decode kernel
    // started, so they are read first; behind the decode kernel the warp
    // then waits for its grid to complete and its writes to be visible
    // (launched on its own, the wait returns at once).
    const int4* entries = p.entries;
    if constexpr (std::is_same<SL, SplitList>::value) {
        if (entries == nullptr) entries = inl.entry;
    }
    RowJob j;
    const bool have = (p.ws_stamp == nullptr || *p.ws_stamp == p.stamp) &&  // this plan's entries
                      locate_row(p, entries, &j);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (have) merge_row(p, j);
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
