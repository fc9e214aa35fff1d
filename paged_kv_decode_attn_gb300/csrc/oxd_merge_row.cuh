// One warp merges the attention states of one output row ("FlashInfer parity
// matrix" page, "Domain coverage": attention state and cascade, state merge).
//
// State i has the log-sum s[i * s_stride] (times s_to_ln it is a natural
// log) and the normalised value row v[i * v_stride + c], c < D:
//   M = max_i s_i, w_i = exp(s_i - M),
//   out = sum_i w_i v_i / sum_i w_i (rounded once to bf16),
//   lse = M + ln sum_i w_i.
// -inf states weigh nothing; a row whose states are all -inf gets out = 0 and
// lse = -inf. Each lane owns 4 consecutive columns; the weighted sum visits
// the states in order. A row of up to 16 states (one pass) is merged with
// every lane holding all the log-sums; longer rows reduce them across the
// warp. A given launch always takes the same path for a row, so results are
// deterministic. Loads go through L2 (ld.global.cg): the states may have been
// written by other CTAs of a still-running grid.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace oxd {

__device__ __forceinline__ uint32_t merge_pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void merge_states_row(const float* s, size_t s_stride, const float* v,
                                                 size_t v_stride, int count, int D,
                                                 float s_to_ln, uint16_t* out_row,
                                                 float* lse_out, int lane) {
    // Values are read kChunk states at a time; the first chunk of a row that
    // fits one 128-column pass is requested together with the log-sums, so
    // a row of up to kChunk states costs one round trip to memory.
    constexpr int kChunk = 16;
    const bool one_pass = D <= 128;
    if (one_pass && count <= kChunk) {
        // Every lane loads all the log-sums (broadcast loads, in the same round
        // trip as the values) and forms the maximum, the weights and their sum
        // itself: no shuffles on the way to the output.
        float sv[kChunk];
        float4 xv[kChunk];
        const bool cols = lane * 4 < D;
#pragma unroll
        for (int i = 0; i < kChunk; ++i) {
            if (i < count) {
                sv[i] = __ldcg(s + static_cast<size_t>(i) * s_stride);
                if (cols)
                    xv[i] = __ldcg(reinterpret_cast<const float4*>(
                        v + static_cast<size_t>(i) * v_stride + lane * 4));
            }
        }
        float M = -INFINITY;
#pragma unroll
        for (int i = 0; i < kChunk; ++i)
            if (i < count) M = fmaxf(M, sv[i] * s_to_ln);
        float W = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) {
#pragma unroll
            for (int i = 0; i < kChunk; ++i) {
                if (i < count) {
                    const float w = expf(sv[i] * s_to_ln - M);
                    W += w;
                    if (cols) {
                        acc.x = fmaf(w, xv[i].x, acc.x);
                        acc.y = fmaf(w, xv[i].y, acc.y);
                        acc.z = fmaf(w, xv[i].z, acc.z);
                        acc.w = fmaf(w, xv[i].w, acc.w);
                    }
                }
            }
        }
        const float inv = W > 0.f ? 1.f / W : 0.f;
        if (cols) {
            uint2 packed;
            packed.x = merge_pack_bf16x2(acc.x * inv, acc.y * inv);
            packed.y = merge_pack_bf16x2(acc.z * inv, acc.w * inv);
            *reinterpret_cast<uint2*>(out_row + lane * 4) = packed;
        }
        if (lane == 0 && lse_out != nullptr) *lse_out = W > 0.f ? M + logf(W) : -INFINITY;
        return;
    }
    // lane i's first log-sum (state i) is loaded once, before the values,
    // and kept for the weights
    const float s_lane =
        lane < count ? __ldcg(s + static_cast<size_t>(lane) * s_stride) * s_to_ln : -INFINITY;
    float4 x[kChunk];
    if (one_pass && lane * 4 < D) {
#pragma unroll
        for (int i = 0; i < kChunk; ++i)
            if (i < count)
                x[i] = __ldcg(reinterpret_cast<const float4*>(v + static_cast<size_t>(i) * v_stride +
                                                              lane * 4));
    }
    // maximum over the states (lanes stride over them), then the sum of
    // weights; with at most 32 states lane i keeps state i's weight
    float M = s_lane;
    for (int i = lane + 32; i < count; i += 32)
        M = fmaxf(M, __ldcg(s + static_cast<size_t>(i) * s_stride) * s_to_ln);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float W = 0.f, w_lane = 0.f;
    if (M != -INFINITY) {
        if (lane < count) {
            w_lane = expf(s_lane - M);
            W = w_lane;
        }
        for (int i = lane + 32; i < count; i += 32)
            W += expf(__ldcg(s + static_cast<size_t>(i) * s_stride) * s_to_ln - M);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    // weighted sum, states in order
    for (int c = lane * 4; c < D; c += 128) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) {
            for (int base = 0; base < count; base += kChunk) {
                if (!(one_pass && base == 0)) {
#pragma unroll
                    for (int i = 0; i < kChunk; ++i)
                        if (base + i < count)
                            x[i] = __ldcg(reinterpret_cast<const float4*>(
                                v + static_cast<size_t>(base + i) * v_stride + c));
                }
#pragma unroll
                for (int i = 0; i < kChunk; ++i) {
                    if (base + i < count) {
                        const int j = base + i;
                        const float w =
                            count <= 32
                                ? __shfl_sync(0xffffffffu, w_lane, j & 31)
                                : expf(__ldcg(s + static_cast<size_t>(j) * s_stride) * s_to_ln - M);
                        acc.x = fmaf(w, x[i].x, acc.x);
                        acc.y = fmaf(w, x[i].y, acc.y);
                        acc.z = fmaf(w, x[i].z, acc.z);
                        acc.w = fmaf(w, x[i].w, acc.w);
                    }
                }
            }
        }
        uint2 packed;
        packed.x = merge_pack_bf16x2(acc.x * inv, acc.y * inv);
        packed.y = merge_pack_bf16x2(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2*>(out_row + c) = packed;
    }
    if (lane == 0 && lse_out != nullptr) *lse_out = W > 0.f ? M + logf(W) : -INFINITY;
}

// The same merge for one half of a 128-column row: columns [64 half, 64 half
// + 64), two per lane, up to 32 states in one pass (the values of 32 states
// take the registers that 16 states of a whole row take). A row of up to 32
// states is merged with every lane holding all the log-sums; longer rows
// reduce them across the warp, with the arithmetic, weights and state order
// merge_states_row uses for them. lse_out is written by the half-0 warp.
__device__ __forceinline__ void merge_states_half_row(const float* s, size_t s_stride,
                                                      const float* v, size_t v_stride, int count,
                                                      float s_to_ln, uint16_t* out_row,
                                                      float* lse_out, int lane, int half) {
    constexpr int kChunk = 32;
    const int c = half * 64 + lane * 2;
    if (count <= kChunk) {
        // One pass: every lane loads all the log-sums (broadcast loads, in the
        // values' round trip) and forms the maximum, the weights and their sum
        // itself, in state order, as merge_states_row does for up to 16 states.
        float sv[kChunk];
        float2 xv[kChunk];
#pragma unroll
        for (int i = 0; i < kChunk; ++i) {
            if (i < count) {
                sv[i] = __ldcg(s + static_cast<size_t>(i) * s_stride);
                xv[i] = __ldcg(reinterpret_cast<const float2*>(v + static_cast<size_t>(i) * v_stride + c));
            }
        }
        float M = -INFINITY;
#pragma unroll
        for (int i = 0; i < kChunk; ++i)
            if (i < count) M = fmaxf(M, sv[i] * s_to_ln);
        float W = 0.f;
        float2 acc = make_float2(0.f, 0.f);
        if (M != -INFINITY) {
#pragma unroll
            for (int i = 0; i < kChunk; ++i) {
                if (i < count) {
                    const float w = expf(sv[i] * s_to_ln - M);
                    W += w;
                    acc.x = fmaf(w, xv[i].x, acc.x);
                    acc.y = fmaf(w, xv[i].y, acc.y);
                }
            }
        }
        const float inv = W > 0.f ? 1.f / W : 0.f;
        *reinterpret_cast<uint32_t*>(out_row + c) = merge_pack_bf16x2(acc.x * inv, acc.y * inv);
        if (half == 0 && lane == 0 && lse_out != nullptr)
            *lse_out = W > 0.f ? M + logf(W) : -INFINITY;
        return;
    }
    const float s_lane =
        lane < count ? __ldcg(s + static_cast<size_t>(lane) * s_stride) * s_to_ln : -INFINITY;
    float2 x[kChunk];
#pragma unroll
    for (int i = 0; i < kChunk; ++i)
        if (i < count)
            x[i] = __ldcg(reinterpret_cast<const float2*>(v + static_cast<size_t>(i) * v_stride + c));
    float M = s_lane;
    for (int i = lane + 32; i < count; i += 32)
        M = fmaxf(M, __ldcg(s + static_cast<size_t>(i) * s_stride) * s_to_ln);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float W = 0.f, w_lane = 0.f;
    if (M != -INFINITY) {
        if (lane < count) {
            w_lane = expf(s_lane - M);
            W = w_lane;
        }
        for (int i = lane + 32; i < count; i += 32)
            W += expf(__ldcg(s + static_cast<size_t>(i) * s_stride) * s_to_ln - M);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    float2 acc = make_float2(0.f, 0.f);
    if (M != -INFINITY) {
        for (int base = 0; base < count; base += kChunk) {
            if (base > 0) {
#pragma unroll
                for (int i = 0; i < kChunk; ++i)
                    if (base + i < count)
                        x[i] = __ldcg(reinterpret_cast<const float2*>(
                            v + static_cast<size_t>(base + i) * v_stride + c));
            }
#pragma unroll
            for (int i = 0; i < kChunk; ++i) {
                if (base + i < count) {
                    const int j = base + i;
                    const float w =
                        count <= 32
                            ? __shfl_sync(0xffffffffu, w_lane, j & 31)
                            : expf(__ldcg(s + static_cast<size_t>(j) * s_stride) * s_to_ln - M);
                    acc.x = fmaf(w, x[i].x, acc.x);
                    acc.y = fmaf(w, x[i].y, acc.y);
                }
            }
        }
    }
    *reinterpret_cast<uint32_t*>(out_row + c) = merge_pack_bf16x2(acc.x * inv, acc.y * inv);
    if (half == 0 && lane == 0 && lse_out != nullptr) *lse_out = W > 0.f ? M + logf(W) : -INFINITY;
}

}  // namespace oxd
