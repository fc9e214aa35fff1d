// Attention-state merge for sm_103a ("FlashInfer parity matrix" page,
// "Domain coverage": attention state and cascade, state merge; and the merge
// step of the "Single decode split-K" row of "Admitted attention matrix").
//
// One warp per output row merges its states with merge_states_row
// (oxd_merge_row.cuh), or, for rows of more than 16 states of 128 columns,
// two warps per row with merge_states_half_row (one pass over up to 32
// states). merge_kernel serves oxd_merge_states (uniform state counts);
// split_merge_kernel the decode and prefill runs' split streams (an entry
// list; launched behind the decode or prefill kernel, it first waits for
// that grid to complete).
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
    int r, count, half;
};

// kHalves warps per output row (1, or 2 for half rows of 128 columns).
template <int kHalves>
__device__ __forceinline__ bool locate_row(const MergeParams& p, const int4* entries, RowJob* j) {
    const long long gw = static_cast<long long>(blockIdx.x) * kWarpsPerBlock + (threadIdx.x >> 5);
    if (gw >= static_cast<long long>(p.n) * p.R * kHalves) return false;
    const long long rw = gw / kHalves;  // row of the warp
    j->half = static_cast<int>(gw - rw * kHalves);
    const int n = static_cast<int>(rw / p.R);
    j->r = static_cast<int>(rw - static_cast<long long>(n) * p.R);
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

template <int kHalves>
__device__ __forceinline__ void merge_row(const MergeParams& p, const RowJob& j) {
    // state i of row r: s[(first + i) * R + r], v[((first + i) * R + r) * D]
    const float* s = p.s + j.first * p.R + j.r;
    const float* v = p.v + (j.first * p.R + j.r) * p.D;
    uint16_t* out = p.out + static_cast<size_t>(j.row0 + j.r) * p.D;
    float* lse = p.lse != nullptr ? p.lse + j.row0 + j.r : nullptr;
    if constexpr (kHalves == 2)
        merge_states_half_row(s, static_cast<size_t>(p.R), v, static_cast<size_t>(p.R) * p.D,
                              j.count, p.s_to_ln, out, lse, threadIdx.x & 31, j.half);
    else
        merge_states_row(s, static_cast<size_t>(p.R), v, static_cast<size_t>(p.R) * p.D, j.count,
                         p.D, p.s_to_ln, out, lse, threadIdx.x & 31);
}

template <int kHalves>
__global__ void __launch_bounds__(kWarpsPerBlock * 32) merge_kernel(const MergeParams p) {
    RowJob j;
    if (locate_row<kHalves>(p, nullptr, &j)) merge_row<kHalves>(p, j);
}

template <class SL, int kHalves>
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
                      locate_row<kHalves>(p, entries, &j);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (have) merge_row<kHalves>(p, j);
}

// Rows of more than 16 states of 128 columns take two warps (one pass each).
int halves_for(const MergeParams& p) {
    return p.D == 128 && (p.uniform ? p.S : p.max_count) > 16 ? 2 : 1;
}

unsigned blocks_for(const MergeParams& p) {
    const long long warps = static_cast<long long>(p.n) * p.R * halves_for(p);
    const long long blocks = (warps + kWarpsPerBlock - 1) / kWarpsPerBlock;
    return blocks > 0x7fffffffLL ? 0u : static_cast<unsigned>(blocks);
}

}  // namespace

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream) {
    const unsigned blocks = blocks_for(p);
    if (blocks == 0) return cudaErrorInvalidConfiguration;
    if (halves_for(p) == 2)
        merge_kernel<2><<<blocks, kWarpsPerBlock * 32, 0, stream>>>(p);
    else
        merge_kernel<1><<<blocks, kWarpsPerBlock * 32, 0, stream>>>(p);
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
    if (halves_for(p) == 2) {
        if (splits != nullptr)
            return cudaLaunchKernelEx(&cfg, split_merge_kernel<SplitList, 2>, p, *splits);
        return cudaLaunchKernelEx(&cfg, split_merge_kernel<NoList, 2>, p, NoList{0});
    }
    if (splits != nullptr)
        return cudaLaunchKernelEx(&cfg, split_merge_kernel<SplitList, 1>, p, *splits);
    return cudaLaunchKernelEx(&cfg, split_merge_kernel<NoList, 1>, p, NoList{0});
}

}  // namespace oxd
