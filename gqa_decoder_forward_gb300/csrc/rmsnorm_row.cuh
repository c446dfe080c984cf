// RMSNorm of one row, shared by the standalone norm kernels and the projections
// that fuse the norm into their prologue, so both give the same bits
// (pull request #1415, section "How": bf16(w * bf16(x * rsqrt(mean(x^2) + eps)))).
//
// mean(x^2) is an fp32 sum in a fixed order over exactly 256 threads: each
// thread sums its elements (8 consecutive per 2048-element stride) in index
// order, a fixed xor-shuffle tree sums each warp, and the eight warp sums are
// added in warp order.  sqrt and the division are IEEE round-to-nearest.
#pragma once

#include "common.cuh"

namespace tfl {

constexpr int kNormThreads = 256;

// 1 / sqrt(mean(x^2) + eps) of row x (H bf16, 16-byte aligned), computed by the
// 256 threads tid = 0..255 of the caller; red holds 8 floats; bar() must
// synchronise exactly those threads.  Every thread returns the same value.
// Rows of up to kRowChunks x 2048 elements are read with every load issued
// before the first sum (one memory round trip); the sums keep the order above.
constexpr int kRowChunks = 4;

// This thread's chunks of row x: chunk j = elements tid*8 + j*2048 .. +7 (zero past H).
__device__ __forceinline__ void load_row_chunks(const bf16* x, int H, int tid, uint4 (&v)[kRowChunks]) {
#pragma unroll
    for (int j = 0; j < kRowChunks; ++j) {
        const int i = tid * 8 + j * kNormThreads * 8;
        v[j] = i < H ? *reinterpret_cast<const uint4*>(x + i) : make_uint4(0u, 0u, 0u, 0u);
    }
}

__device__ __forceinline__ float sumsq_chunks(const uint4 (&v)[kRowChunks], int H, int tid) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < kRowChunks; ++j) {
        if (tid * 8 + j * kNormThreads * 8 >= H) break;
        const bf16* e = reinterpret_cast<const bf16*>(&v[j]);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float f = bf(e[k]);
            ss = fmaf(f, f, ss);
        }
    }
    return ss;
}

// Block part of rms_inv: this thread's sum ss -> 1 / sqrt(mean + eps).
template <typename Barrier>
__device__ __forceinline__ float rms_finish(float ss, int H, float eps, int tid, float* red, Barrier bar) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    bar();
    float s = red[0];
#pragma unroll
    for (int w = 1; w < kNormThreads / 32; ++w) s += red[w];
    return 1.0f / sqrtf(s / (float)H + eps);
}

template <typename Barrier>
__device__ __forceinline__ float rms_inv(const bf16* x, int H, float eps, int tid, float* red, Barrier bar) {
    float ss = 0.f;
    if (H <= kRowChunks * kNormThreads * 8) {
        uint4 v[kRowChunks];
        load_row_chunks(x, H, tid, v);
        ss = sumsq_chunks(v, H, tid);
    } else {
        for (int i = tid * 8; i < H; i += kNormThreads * 8) {
            uint4 v = *reinterpret_cast<const uint4*>(x + i);
            const bf16* e = reinterpret_cast<const bf16*>(&v);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                float f = bf(e[k]);
                ss = fmaf(f, f, ss);
            }
        }
    }
    return rms_finish(ss, H, eps, tid, red, bar);
}

// The normalised element: bf16(w * bf16(x * r)).
__device__ __forceinline__ bf16 rms_apply(bf16 x, bf16 w, float r) { return rn(bf(w) * rbf(bf(x) * r)); }

}  // namespace tfl
