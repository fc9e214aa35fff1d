// Host-side helpers shared by the library's C-ABI files: spans, overlap and
// alignment checks, and the entry points into oxd_host.cpp's tensor-map
// encoder, plan stamps and run epochs. Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <stddef.h>
#include <stdint.h>

namespace oxd {

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Span {
    uintptr_t lo, hi;  // [lo, hi)
};

inline Span span(const void* p, size_t bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return {a, a + bytes};
}

inline bool overlap(const Span& a, const Span& b) {
    return a.lo < a.hi && b.lo < b.hi && a.lo < b.hi && b.lo < a.hi;
}

// 4-D map over a K or V pool: (d, A, B, page) with (A, B) = (head, token)
// for NHD and (token, head) for HND; a box is 64 columns x all page_size
// tokens of one head, stored with the 128-byte swizzle.
bool encode_kv_pool(CUtensorMap* map, const void* pool, int layout, int page_size,
                    int num_kv_heads, int64_t num_pages);
// bf16 tensor map of `rank` dimensions (dims innermost first, byte strides of
// dims 1..rank-1), 128-byte swizzle, zero fill past the edges.
bool encode_bf16_map(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides, const uint32_t* box);
// Plan stamps: never 0, unique within the process, random across processes.
unsigned long long next_plan_stamp();

}  // namespace oxd
