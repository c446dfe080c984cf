// Decode attention: causal GQA of a few rows per stream over a position-major
// paged bf16 cache, split over key blocks at absolute positions (pull request
// #1415, section "How": "decode rows on sdpa_vector lanes over key blocks at
// absolute positions").
//
// Pass 1 (attn_block_kernel): one CTA per (key block b of 128 positions, KV
// head g, group of <= 4 rows of one stream).  The block's keys and values for
// head g are staged in shared memory with cp.async, the G = n_q/n_kv query
// heads of each row read them, and the CTA writes per (row, head) the block's
// max score m_b, sum l_b = sum exp(s - m_b) and o_b = sum exp(s - m_b) v.
// Pass 2 (attn_merge_kernel): per (row, head), M = max_b m_b, then
// L = sum_b l_b e^(m_b - M) and O = sum_b o_b e^(m_b - M) in block order,
// out = bf16(O / L).
//
// Scores are fp32 dot products in d order of q (pre-scaled by log2(e)/sqrt(D))
// with the bf16 keys; softmax weights stay fp32 (never rounded to bf16).
// Every row's arithmetic depends only on its own position: the block split is
// fixed by absolute position and masked keys contribute exact zeros, so a row
// gives the same bits alone or beside other rows (one-row steps == windows).
#include "common.cuh"

namespace tfl {
namespace {

constexpr int kThreads = 256;
constexpr int kRB = 4;          // rows per CTA
constexpr int kKB = kPage;      // keys per block
constexpr int kKPad = kHeadDim + 8;  // padded key row in shared memory (bf16)
constexpr int kMaxG = 8;        // query heads per KV head
constexpr int kMaxPairs = kRB * kMaxG;

struct Smem {
    float q[kMaxPairs][kHeadDim];          // 16 KB
    float s[kMaxPairs][kKB];               // 16 KB scores, then weights
    union {
        bf16 k[kKB][kKPad];                // 34 KB
        float red[2][kMaxPairs][kHeadDim]; // 32 KB (after the scores)
    } u;
    bf16 v[kKB][kHeadDim];                 // 32 KB
    float m[kMaxPairs];
    float l[kMaxPairs];
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    unsigned sa = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem));
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Locates row group z: stream s, first row (global index) r0, row count nr.
__device__ __forceinline__ bool find_group(const RowMap& m, int z, int& s, int& r0, int& nr) {
    for (int t = 0; t < m.n_streams; ++t) {
        int rows = m.row_start[t + 1] - m.row_start[t];
        int ng = (rows + kRB - 1) / kRB;
        if (z < ng) {
            s = t;
            r0 = m.row_start[t] + z * kRB;
            nr = min(kRB, rows - z * kRB);
            return true;
        }
        z -= ng;
    }
    return false;
}

// G = query heads per KV head (compile-time, so every per-pair loop has a fixed
// length and the accumulators stay in registers).
template <int G>
__global__ void __launch_bounds__(kThreads, 2) attn_block_kernel(const __grid_constant__ AttnDecodeArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
    pdl_wait();

    int s, r0, nr;
    if (!find_group(a.rows, blockIdx.z, s, r0, nr)) return;
    const int b = blockIdx.x, g = blockIdx.y;
    const int p_first = a.rows.pos0[s] + (r0 - a.rows.row_start[s]);
    const int p_last = p_first + nr - 1;
    const int k0 = b * kKB;
    if (k0 > p_last) return;
    const int nv = min(kKB, p_last + 1 - k0);  // keys of this block any row sees
    const int tid = threadIdx.x;

    // stage keys and values of head g (rows of 256 B inside one page)
    const KvView& kv = a.rows.kv[s];
    const bf16* kbase = kv_row(kv, a.layer, 0, k0, a.n_kv) + (size_t)g * kHeadDim;
    const bf16* vbase = kv_row(kv, a.layer, 1, k0, a.n_kv) + (size_t)g * kHeadDim;
    const size_t pstride = (size_t)a.n_kv * kHeadDim;
    for (int i = tid; i < nv * 16; i += kThreads) {
        int t = i >> 4, c = i & 15;
        cp_async16(&sm.u.k[t][c * 8], kbase + t * pstride + c * 8);
        cp_async16(&sm.v[t][c * 8], vbase + t * pstride + c * 8);
    }
    // queries, pre-scaled: pair p = i*G + hh (row i of the group, head g*G + hh)
    const int P = nr * G;
    const float qscale = 1.4426950408889634f * rsqrtf((float)kHeadDim);
    for (int i = tid; i < P * kHeadDim; i += kThreads) {
        int p = i / kHeadDim, d = i % kHeadDim;
        int row = r0 + p / G, head = g * G + p % G;
        sm.q[p][d] = bf(a.q[(size_t)row * a.n_q * kHeadDim + (size_t)head * kHeadDim + d]) * qscale;
    }
    cp_async_wait_all();
    __syncthreads();

    // scores: thread -> key t; the two thread halves split the G heads
    {
        constexpr int GH = (G + 1) / 2;
        const int t = tid & (kKB - 1), half = tid >> 7;
        const int h0 = half * GH, hn = half ? G - GH : GH;
        float acc[kRB][GH];
#pragma unroll
        for (int i = 0; i < kRB; ++i)
#pragma unroll
            for (int j = 0; j < GH; ++j) acc[i][j] = 0.f;
        if (t < nv) {
#pragma unroll 2
            for (int d = 0; d < kHeadDim; d += 8) {
                uint4 kw = *reinterpret_cast<const uint4*>(&sm.u.k[t][d]);
                const bf16* kk = reinterpret_cast<const bf16*>(&kw);
                float kf[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) kf[e] = bf(kk[e]);
#pragma unroll
                for (int i = 0; i < kRB; ++i) {
                    if (i < nr) {
#pragma unroll
                        for (int j = 0; j < GH; ++j) {
                            if (j < hn) {
                                const float* qq = &sm.q[i * G + h0 + j][d];
#pragma unroll
                                for (int e = 0; e < 8; ++e) acc[i][j] = fmaf(qq[e], kf[e], acc[i][j]);
                            }
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kRB; ++i) {
            if (i < nr) {
                const bool vis = t < nv && k0 + t <= p_first + i;
#pragma unroll
                for (int j = 0; j < GH; ++j)
                    if (j < hn) sm.s[i * G + h0 + j][t] = vis ? acc[i][j] : -INFINITY;
            }
        }
    }
    __syncthreads();

    // softmax statistics of the block: warp per pair, lane per 4 keys
    {
        const int warp = tid >> 5, lane = tid & 31;
        for (int p = warp; p < P; p += kThreads / 32) {
            float x0 = sm.s[p][lane * 4 + 0], x1 = sm.s[p][lane * 4 + 1];
            float x2 = sm.s[p][lane * 4 + 2], x3 = sm.s[p][lane * 4 + 3];
            float m = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            float e0 = 0.f, e1 = 0.f, e2 = 0.f, e3 = 0.f;
            if (m != -INFINITY) {
                e0 = exp2f(x0 - m);
                e1 = exp2f(x1 - m);
                e2 = exp2f(x2 - m);
                e3 = exp2f(x3 - m);
            }
            float l = ((e0 + e1) + e2) + e3;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
            sm.s[p][lane * 4 + 0] = e0;
            sm.s[p][lane * 4 + 1] = e1;
            sm.s[p][lane * 4 + 2] = e2;
            sm.s[p][lane * 4 + 3] = e3;
            if (lane == 0) {
                sm.m[p] = m;
                sm.l[p] = l;
            }
        }
    }
    __syncthreads();

    // P.V: thread -> dim d, half of the keys; halves added in order
    {
        const int d = tid & (kHeadDim - 1), half = tid >> 7;
        const int tb = half * (kKB / 2), te = min(nv, tb + kKB / 2);
        float acc[kRB][G];
#pragma unroll
        for (int i = 0; i < kRB; ++i)
#pragma unroll
            for (int j = 0; j < G; ++j) acc[i][j] = 0.f;
        for (int t = tb; t < te; ++t) {
            const float vv = bf(sm.v[t][d]);
#pragma unroll
            for (int i = 0; i < kRB; ++i) {
                if (i < nr) {
#pragma unroll
                    for (int j = 0; j < G; ++j) {
                        // a zero weight (a masked key) leaves the sum untouched, even its sign
                        const float w = sm.s[i * G + j][t];
                        if (w != 0.f) acc[i][j] = fmaf(w, vv, acc[i][j]);
                    }
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kRB; ++i)
            if (i < nr)
#pragma unroll
                for (int j = 0; j < G; ++j) sm.u.red[half][i * G + j][d] = acc[i][j];
    }
    __syncthreads();
    pdl_trigger();

    for (int i = tid; i < P * kHeadDim; i += kThreads) {
        const int p = i / kHeadDim, d = i % kHeadDim;
        const int row = r0 + p / G, head = g * G + p % G;
        const size_t idx = ((size_t)row * a.n_q + head) * a.max_blocks + b;
        a.po[idx * kHeadDim + d] = sm.u.red[0][p][d] + sm.u.red[1][p][d];
        if (d == 0) {
            a.pm[idx] = sm.m[p];
            a.pl[idx] = sm.l[p];
        }
    }
}

__global__ void __launch_bounds__(kHeadDim) attn_merge_kernel(const __grid_constant__ AttnDecodeArgs a) {
    __shared__ float wts[1024];
    __shared__ float red[kHeadDim / 32];
    pdl_wait();
    const int head = blockIdx.x, row = blockIdx.y, d = threadIdx.x;
    const int s = row_stream(a.rows, row);
    const int pos = a.rows.pos0[s] + (row - a.rows.row_start[s]);
    const int nb = pos / kKB + 1;
    const size_t base = ((size_t)row * a.n_q + head) * a.max_blocks;

    float M = -INFINITY;
    for (int b = d; b < nb; b += kHeadDim) M = fmaxf(M, a.pm[base + b]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if ((d & 31) == 0) red[d >> 5] = M;
    __syncthreads();
    M = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));

    float O = 0.f, L = 0.f;
    for (int c = 0; c < nb; c += 1024) {
        const int n = min(1024, nb - c);
        __syncthreads();
        for (int b = d; b < n; b += kHeadDim) wts[b] = exp2f(a.pm[base + c + b] - M);
        __syncthreads();
#pragma unroll 8
        for (int b = 0; b < n; ++b) {
            const float w = wts[b];
            L = fmaf(a.pl[base + c + b], w, L);
            O = fmaf(a.po[(base + c + b) * kHeadDim + d], w, O);
        }
    }
    pdl_trigger();
    a.out[(size_t)row * a.n_q * kHeadDim + (size_t)head * kHeadDim + d] = rn(O / L);
}

}  // namespace

cudaError_t init_attn_decode() {
    cudaError_t e = cudaFuncSetAttribute(attn_block_kernel<7>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sizeof(Smem));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(attn_block_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(Smem));
}

int attn_decode_blocks(const AttnDecodeArgs& a, int* groups) {
    int g = 0, max_pos = 0;
    for (int s = 0; s < a.rows.n_streams; ++s) {
        int rows = a.rows.row_start[s + 1] - a.rows.row_start[s];
        g += (rows + kRB - 1) / kRB;
        max_pos = max(max_pos, a.rows.pos0[s] + rows - 1);
    }
    *groups = g;
    return max_pos / kKB + 1;
}

cudaError_t launch_attn_block(const AttnDecodeArgs& a, cudaStream_t st, bool pdl) {
    const int G = a.n_q / a.n_kv;
    if ((G != 7 && G != 8) || a.n_q % a.n_kv != 0) return cudaErrorInvalidValue;
    int groups = 0;
    const int nblk = attn_decode_blocks(a, &groups);
    if (nblk > a.max_blocks) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t c1 = {};
    c1.gridDim = dim3(nblk, a.n_kv, groups);
    c1.blockDim = dim3(kThreads);
    c1.dynamicSmemBytes = (int)sizeof(Smem);
    c1.stream = st;
    c1.attrs = attr;
    c1.numAttrs = pdl ? 1 : 0;
    return G == 7 ? cudaLaunchKernelEx(&c1, attn_block_kernel<7>, a) : cudaLaunchKernelEx(&c1, attn_block_kernel<8>, a);
}

cudaError_t launch_attn_merge(const AttnDecodeArgs& a, cudaStream_t st, bool pdl) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t c2 = {};
    c2.gridDim = dim3(a.n_q, a.rows.n_rows);
    c2.blockDim = dim3(kHeadDim);
    c2.stream = st;
    c2.attrs = attr;
    c2.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&c2, attn_merge_kernel, a);
}

}  // namespace tfl
