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
template <typename Barrier>
__device__ __forceinline__ float rms_inv(const bf16* x, int H, float eps, int tid, float* red, Barrier bar) {
    float ss = 0.f;
    for (int i = tid * 8; i < H; i += kNormThreads * 8) {
        uint4 v = *reinterpret_cast<const uint4*>(x + i);
        const bf16* e = reinterpret_cast<const bf16*>(&v);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            float f = bf(e[k]);
            ss = fmaf(f, f, ss);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    bar();
    float s = red[0];
#pragma unroll
    for (int w = 1; w < kNormThreads / 32; ++w) s += red[w];
    return 1.0f / sqrtf(s / (float)H + eps);
}

// The normalised element: bf16(w * bf16(x * r)).
__device__ __forceinline__ bf16 rms_apply(bf16 x, bf16 w, float r) { return rn(bf(w) * rbf(bf(x) * r)); }

}  // namespace tfl
