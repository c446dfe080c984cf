// Per-row kernels: embedding gather, RMSNorm, vocabulary argmax, KV copies.
//
// RMSNorm (pull request #1415, section "How"):
//   out = bf16(w * bf16(x * r)),  r = 1 / sqrt(mean(x^2) + eps)
// mean(x^2) is an fp32 sum in a fixed order (per thread in index order, then a
// fixed shuffle tree, then warps in order), so a row's result does not depend
// on how many rows share the launch.  sqrt and the divisions are the IEEE
// round-to-nearest operations (no fast-math approximations).
//
// Argmax (same pull request, teacher-forced misses reply: "Both sides break
// ties to the lower id"; its teacher-forced checks refuse rows holding NaN or +-Inf): the
// largest logit, the lowest id among equal maxima; a row with any non-finite
// logit yields -1 and raises a bit of the device status word.
#include "common.cuh"
#include "rmsnorm_row.cuh"

namespace tfl {
namespace {

// x: the row (H bf16, 16-byte aligned); writes the normalised row to out.
__device__ __forceinline__ void rmsnorm_row(const bf16* x, const bf16* w, float eps, int H, bf16* out, float* red) {
    const float r = rms_inv(x, H, eps, threadIdx.x, red, [] { __syncthreads(); });
    for (int i = threadIdx.x * 8; i < H; i += kNormThreads * 8) {
        uint4 v = *reinterpret_cast<const uint4*>(x + i);
        uint4 wv = __ldg(reinterpret_cast<const uint4*>(w + i));
        const bf16* e = reinterpret_cast<const bf16*>(&v);
        const bf16* we = reinterpret_cast<const bf16*>(&wv);
        uint4 o;
        bf16* oe = reinterpret_cast<bf16*>(&o);
#pragma unroll
        for (int k = 0; k < 8; ++k) oe[k] = rms_apply(e[k], we[k], r);
        *reinterpret_cast<uint4*>(out + i) = o;
    }
}

__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(const bf16* x, const bf16* w, float eps, int H,
                                                              bf16* out) {
    __shared__ float red[kNormThreads / 32];
    pdl_wait();
    pdl_trigger();
    const size_t row = blockIdx.x;
    rmsnorm_row(x + row * H, w, eps, H, out + row * H, red);
}

__global__ void __launch_bounds__(kNormThreads) embed_rmsnorm_kernel(const int32_t* ids, const bf16* embed, int vocab,
                                                                    const bf16* w, float eps, int H, bf16* h, bf16* xn,
                                                                    int* status) {
    __shared__ float red[kNormThreads / 32];
    pdl_wait();
    pdl_trigger();
    const size_t row = blockIdx.x;
    const int id = ids[row];
    bf16* hr = h + row * H;
    if (id < 0 || id >= vocab) {
        for (int i = threadIdx.x * 8; i < H; i += kNormThreads * 8)
            *reinterpret_cast<uint4*>(hr + i) = make_uint4(0u, 0u, 0u, 0u);
        if (threadIdx.x == 0) atomicOr(status, kStatusBadToken);
    } else {
        const bf16* er = embed + (size_t)id * H;
        for (int i = threadIdx.x * 8; i < H; i += kNormThreads * 8)
            *reinterpret_cast<uint4*>(hr + i) = __ldg(reinterpret_cast<const uint4*>(er + i));
    }
    __syncthreads();
    rmsnorm_row(hr, w, eps, H, xn + row * H, red);
}

constexpr int kArgThreads = 1024;

__global__ void __launch_bounds__(kArgThreads) argmax_kernel(const bf16* logits, int V, int32_t* ids, int* status,
                                                              int bad_id) {
    __shared__ float bv[kArgThreads / 32];
    __shared__ int bi[kArgThreads / 32];
    __shared__ int bad_any;
    pdl_wait();
    pdl_trigger();
    if (threadIdx.x == 0) bad_any = 0;
    __syncthreads();
    const bf16* row = logits + (size_t)blockIdx.x * V;
    float best = -INFINITY;
    int idx = 0x7fffffff;
    bool bad = false;
    for (int i = threadIdx.x * 8; i < V; i += kArgThreads * 8) {
        uint4 v = __ldg(reinterpret_cast<const uint4*>(row + i));
        const bf16* e = reinterpret_cast<const bf16*>(&v);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            float f = bf(e[k]);
            if (!isfinite(f)) bad = true;
            else if (f > best) { best = f; idx = i + k; }  // ascending ids: ties keep the lower
        }
    }
    if (bad) bad_any = 1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, best, o);
        int oi = __shfl_xor_sync(0xffffffffu, idx, o);
        if (ov > best || (ov == best && oi < idx)) { best = ov; idx = oi; }
    }
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) { bv[warp] = best; bi[warp] = idx; }
    __syncthreads();
    if (threadIdx.x == 0) {
        float b = bv[0];
        int j = bi[0];
        for (int w = 1; w < kArgThreads / 32; ++w)
            if (bv[w] > b || (bv[w] == b && bi[w] < j)) { b = bv[w]; j = bi[w]; }
        if (bad_any) {
            ids[blockIdx.x] = bad_id;
            atomicOr(status, kStatusNonFinite);
        } else {
            ids[blockIdx.x] = j;
        }
    }
}

// One CTA per position: copies the n_kv*D keys and values of (layer, pos0 + i).
__global__ void kv_copy_kernel(KvView kv, int n_kv, int layer, int pos0, bf16* k, bf16* v, int to_cache) {
    const int i = blockIdx.x;
    const int pos = pos0 + i;
    const int w = n_kv * kHeadDim;
    bf16* kc = kv_row(kv, layer, 0, pos, n_kv);
    bf16* vc = kv_row(kv, layer, 1, pos, n_kv);
    bf16* kd = k + (size_t)i * w;
    bf16* vd = v + (size_t)i * w;
    for (int j = threadIdx.x * 8; j < w; j += blockDim.x * 8) {
        if (to_cache) {
            *reinterpret_cast<uint4*>(kc + j) = *reinterpret_cast<const uint4*>(kd + j);
            *reinterpret_cast<uint4*>(vc + j) = *reinterpret_cast<const uint4*>(vd + j);
        } else {
            *reinterpret_cast<uint4*>(kd + j) = *reinterpret_cast<const uint4*>(kc + j);
            *reinterpret_cast<uint4*>(vd + j) = *reinterpret_cast<const uint4*>(vc + j);
        }
    }
}

cudaLaunchConfig_t row_cfg(int rows, int threads, cudaStream_t st, cudaLaunchAttribute* attr, bool pdl) {
    cudaLaunchConfig_t c = {};
    c.gridDim = dim3(rows);
    c.blockDim = dim3(threads);
    c.stream = st;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    c.attrs = attr;
    c.numAttrs = pdl ? 1 : 0;
    return c;
}

}  // namespace

cudaError_t launch_rmsnorm(const bf16* x, const bf16* w, float eps, int n_rows, int H, bf16* out, cudaStream_t st,
                           bool pdl) {
    if (H % 8 != 0 || n_rows < 1) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t c = row_cfg(n_rows, kNormThreads, st, attr, pdl);
    return cudaLaunchKernelEx(&c, rmsnorm_kernel, x, w, eps, H, out);
}

cudaError_t launch_embed_rmsnorm(const int32_t* ids, const bf16* embed, int vocab, const bf16* w, float eps,
                                 int n_rows, int H, bf16* h, bf16* xn, int* status, cudaStream_t st, bool pdl) {
    if (H % 8 != 0 || n_rows < 1) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t c = row_cfg(n_rows, kNormThreads, st, attr, pdl);
    return cudaLaunchKernelEx(&c, embed_rmsnorm_kernel, ids, embed, vocab, w, eps, H, h, xn, status);
}

cudaError_t launch_argmax(const bf16* logits, int n_rows, int V, int32_t* ids, int* status, cudaStream_t st,
                          bool pdl, int bad_id) {
    if (V % 8 != 0 || n_rows < 1) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t c = row_cfg(n_rows, kArgThreads, st, attr, pdl);
    return cudaLaunchKernelEx(&c, argmax_kernel, logits, V, ids, status, bad_id);
}

cudaError_t launch_kv_copy(bf16* pages, const int* table, int n_pages, int n_kv, int layer, int pos0, int n, bf16* k,
                           bf16* v, bool to_cache, cudaStream_t st) {
    if (n < 1) return cudaSuccess;
    KvView kv;
    kv.pages = pages;
    kv.table = table;
    kv.n_pages = n_pages;
    kv.pad_ = 0;
    kv_copy_kernel<<<n, 128, 0, st>>>(kv, n_kv, layer, pos0, k, v, to_cache ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace tfl
