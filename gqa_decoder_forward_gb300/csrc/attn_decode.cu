// Decode attention: causal GQA of a few rows per stream over a position-major
// paged bf16 cache, split over key blocks at absolute positions (pull request
// #1415, section "How": "decode rows on sdpa_vector lanes over key blocks at
// absolute positions").
//
// Pass 1 (attn_block_kernel): one CTA per (key block b of 128 positions, KV
// head g, group of <= 4 rows of one stream).  The block's keys and values for
// head g are staged in shared memory with cp.async.  The G = n_q/n_kv query
// heads of the group's rows form the M dimension of tensor-core products
// (mma.sync m16n8k16, bf16 in, fp32 accumulate): S = Q K^T over the 128 keys,
// then O = P V.  Per (row, head) the CTA writes the block's max score m_b, sum
// l_b = sum exp(s - m_b) and o_b = sum exp(s - m_b) v.
// Pass 2 (attn_merge_kernel): per (row, head), M = max_b m_b, then
// L = sum_b l_b e^(m_b - M) and O = sum_b o_b e^(m_b - M) in block order,
// out = bf16(O / L).
//
// Precision: scores are fp32 dot products of the bf16 q and k, scaled in fp32;
// softmax weights are fp32 and enter P V as a pair of bf16 numbers
// (hi = bf16(p), lo = bf16(p - hi)), i.e. with about 16 significant bits --
// the weights are not rounded to bf16.
//
// Determinism: every row's arithmetic depends only on its own position: the
// block split is fixed by absolute position, masked keys have weight exactly
// 0, keys past the last one any row of the group sees are zero-filled in
// shared memory, and each output element of an mma depends only on its own
// row of P.  A row gives the same bits alone or beside other rows (one-row
// steps == windows, solo == batched).
#include "common.cuh"
#include "warp_mma.cuh"

namespace tfl {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRB = 4;               // rows per CTA
constexpr int kKB = kPage;           // keys per block
constexpr int kMaxPairs = 32;        // kRB rows x up to 8 heads, two m16 tiles
constexpr int kMergeSlices = 8;      // block slices of one merge CTA

// Rows of 128 bf16 (256 bytes, 16 chunks of 16 bytes) with chunk c of row r
// stored at chunk c ^ (r & 7): the eight rows an ldmatrix reads hit distinct
// banks without padding.
__device__ __forceinline__ int swz(int row, int col) {
    return row * kHeadDim + (((col >> 3) ^ (row & 7)) << 3) + (col & 7);
}

// 75,776 bytes: three CTAs per SM.  The softmax weights (hi and lo parts,
// 2 x 32 x 128 bf16) reuse the key tile once the scores are computed.
struct Smem {
    bf16 q[kMaxPairs * kHeadDim];    // 8 KB
    bf16 k[kKB * kHeadDim];          // 32 KB (then the weights)
    bf16 v[kKB * kHeadDim];          // 32 KB
    float wmax[kWarps][kMaxPairs];   // per-warp row maxima
    float wsum[kWarps][kMaxPairs];   // per-warp row sums
};

using wm::cp_async16_zfill;
using wm::cp_async_commit;
using wm::cp_async_wait;
using wm::ldsm_x4;
using wm::ldsm_x4_t;
using wm::mma16816;
using wm::pack_bf16;

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

// G = query heads per KV head.  Pair p = i*G + j is (row i of the group, head g*G + j).
template <int G>
__global__ void __launch_bounds__(kThreads, 3) attn_block_kernel(const __grid_constant__ AttnDecodeArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>(smem_raw);

    int s, r0, nr;
    if (!find_group(a.rows, blockIdx.z, s, r0, nr)) return;
    const int b = blockIdx.x, g = blockIdx.y;
    const int p_first = a.rows.pos0[s] + (r0 - a.rows.row_start[s]);
    const int p_last = p_first + nr - 1;
    const int k0 = b * kKB;
    if (k0 > p_last) return;
    const int nv = min(kKB, p_last + 1 - k0);  // keys of this block any row sees
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, tig = lane & 3;
    const int P = nr * G;
    const int MT = (P + 15) / 16;  // m16 tiles of pairs

    // stage keys and values of head g (rows of 256 B inside one page); keys past
    // nv are zero-filled so that their weight-0 products stay exact zeros.  Keys
    // first, values second, as two copy groups.
    const KvView& kv = a.rows.kv[s];
    const bf16* kbase = kv_row(kv, a.layer, 0, k0, a.n_kv) + (size_t)g * kHeadDim;
    const bf16* vbase = kv_row(kv, a.layer, 1, k0, a.n_kv) + (size_t)g * kHeadDim;
    const size_t pstride = (size_t)a.n_kv * kHeadDim;
    auto stage = [&](bf16* dst, const bf16* src) {
        for (int i = tid; i < kKB * 16; i += kThreads) {
            const int t = i >> 4, c = i & 15;
            const bool valid = t < nv;
            cp_async16_zfill(dst + swz(t, c * 8), src + (valid ? t * pstride + c * 8 : 0), valid);
        }
        cp_async_commit();
    };
    // A block whose keys all precede the stream's first row of this call holds
    // cache rows written by earlier calls (every kernel of the library signals
    // its dependents only after its own dependency wait, so those writers have
    // completed): it streams in while the previous kernel is still finishing.
    const bool early = k0 + nv <= a.rows.pos0[s];
    if (early) {
        stage(sm.k, kbase);
        stage(sm.v, vbase);
    }
    pdl_wait();
    pdl_trigger();
    if (!early) {
        stage(sm.k, kbase);
        stage(sm.v, vbase);
    }
    // queries (bf16, unscaled); pairs past P are zero
    for (int i = tid; i < MT * 16 * 16; i += kThreads) {
        const int p = i >> 4, c = i & 15;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (p < P) {
            const int row = r0 + p / G, head = g * G + p % G;
            val = *reinterpret_cast<const uint4*>(a.q + (size_t)row * a.n_q * kHeadDim + (size_t)head * kHeadDim +
                                                   c * 8);
        }
        *reinterpret_cast<uint4*>(&sm.q[swz(p, c * 8)]) = val;
    }
    cp_async_wait<1>();  // the keys have landed; the values may still be in flight
    __syncthreads();

    // ---- S = Q K^T: warp w owns keys 16w .. 16w+15 (two n8 tiles) ----
    const float kScale = 0.12751743074640502f;  // log2(e) / sqrt(128)
    float sc[2][2][4];  // [m tile][n tile][fragment]
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) sc[mt][nt][0] = sc[mt][nt][1] = sc[mt][nt][2] = sc[mt][nt][3] = 0.f;
    {
        const int mrow = (lane & 7) + ((lane >> 3) & 1) * 8, mcol = (lane >> 4) * 8;     // A: matrices (r, k) quads
        const int krow = (lane & 7) + (lane >> 4) * 8, kcol = ((lane >> 3) & 1) * 8;     // B: keys x dims
#pragma unroll
        for (int ks = 0; ks < kHeadDim / 16; ++ks) {
            uint32_t bk[4];
            ldsm_x4(bk, &sm.k[swz(warp * 16 + krow, ks * 16 + kcol)]);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                if (mt < MT) {
                    uint32_t aq[4];
                    ldsm_x4(aq, &sm.q[swz(mt * 16 + mrow, ks * 16 + mcol)]);
                    mma16816(sc[mt][0], aq, bk[0], bk[1]);
                    mma16816(sc[mt][1], aq, bk[2], bk[3]);
                }
            }
        }
    }
    // scale, mask, per-warp row maxima
    float mx[2][2];  // [m tile][row half]
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int p = mt * 16 + gq + h * 8;
            const int pos_row = p_first + (p < P ? p / G : 0);
            float m = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int t = warp * 16 + nt * 8 + 2 * tig + e;
                    const bool vis = p < P && t < nv && k0 + t <= pos_row;
                    float& v = sc[mt][nt][h * 2 + e];
                    v = vis ? v * kScale : -INFINITY;
                    m = fmaxf(m, v);
                }
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            mx[mt][h] = m;
        }
    }
    if (tig == 0) {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h) sm.wmax[warp][mt * 16 + gq + h * 8] = mx[mt][h];
    }
    __syncthreads();
    // block row maxima, weights, per-warp row sums, weights to shared memory
    // (over the key tile, which no warp reads any more)
    bf16* pw = sm.k;
    float bmax[2][2];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int p = mt * 16 + gq + h * 8;
            float m = sm.wmax[0][p];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) m = fmaxf(m, sm.wmax[w][p]);
            bmax[mt][h] = m;
            float l = 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                float e0 = 0.f, e1 = 0.f;
                if (m != -INFINITY) {
                    e0 = exp2f(sc[mt][nt][h * 2 + 0] - m);
                    e1 = exp2f(sc[mt][nt][h * 2 + 1] - m);
                }
                l += e0;
                l += e1;
                const bf16 h0 = rn(e0), h1 = rn(e1);
                const bf16 l0 = rn(e0 - bf(h0)), l1 = rn(e1 - bf(h1));
                const int t = warp * 16 + nt * 8 + 2 * tig;
                *reinterpret_cast<uint32_t*>(&pw[swz(p, t)]) = pack_bf16(h0, h1);
                *reinterpret_cast<uint32_t*>(&pw[kMaxPairs * kHeadDim + swz(p, t)]) = pack_bf16(l0, l1);
            }
            l += __shfl_xor_sync(0xffffffffu, l, 1);
            l += __shfl_xor_sync(0xffffffffu, l, 2);
            if (tig == 0) sm.wsum[warp][p] = l;
        }
    }
    cp_async_wait<0>();  // the values
    __syncthreads();

    // ---- O = P V: warp w owns dims 16w .. 16w+15 (two n8 tiles) ----
    float oc[2][2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) oc[mt][nt][0] = oc[mt][nt][1] = oc[mt][nt][2] = oc[mt][nt][3] = 0.f;
    {
        const int mrow = (lane & 7) + ((lane >> 3) & 1) * 8, mcol = (lane >> 4) * 8;  // A: pairs x keys
        const int vrow = (lane & 7) + ((lane >> 3) & 1) * 8, vcol = (lane >> 4) * 8;  // B (trans): keys x dims
#pragma unroll 2
        for (int ks = 0; ks < kKB / 16; ++ks) {
            uint32_t bv[4];
            ldsm_x4_t(bv, &sm.v[swz(ks * 16 + vrow, warp * 16 + vcol)]);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                if (mt < MT) {
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
                        uint32_t ap[4];
                        ldsm_x4(ap, &pw[part * kMaxPairs * kHeadDim + swz(mt * 16 + mrow, ks * 16 + mcol)]);
                        mma16816(oc[mt][0], ap, bv[0], bv[1]);
                        mma16816(oc[mt][1], ap, bv[2], bv[3]);
                    }
                }
            }
        }
    }

    // ---- partials: o (unnormalised), m, l per (row, head) ----
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int p = mt * 16 + gq + h * 8;
            if (mt < MT && p < P) {
                const int row = r0 + p / G, head = g * G + p % G;
                const size_t idx = ((size_t)row * a.n_q + head) * a.max_blocks + b;
                float* po = a.po + idx * kHeadDim + warp * 16 + 2 * tig;
                *reinterpret_cast<float2*>(po) = make_float2(oc[mt][0][h * 2 + 0], oc[mt][0][h * 2 + 1]);
                *reinterpret_cast<float2*>(po + 8) = make_float2(oc[mt][1][h * 2 + 0], oc[mt][1][h * 2 + 1]);
                if (warp == 0 && tig == 0) {
                    float l = sm.wsum[0][p];
#pragma unroll
                    for (int w = 1; w < kWarps; ++w) l += sm.wsum[w][p];
                    a.pm[idx] = bmax[mt][h];
                    a.pl[idx] = l;
                }
            }
        }
    }
}

// One CTA per (head, row), kMergeSlices x 128 threads: thread (slice i, dim d)
// folds blocks i, i + 8, i + 16, ... in order, all its loads issued ahead; the
// eight slice sums are then added in slice order.  The fold depends only on
// the row's position (its block count), never on the other rows of the call.
__global__ void __launch_bounds__(kHeadDim* kMergeSlices) attn_merge_kernel(const __grid_constant__ AttnDecodeArgs a) {
    constexpr int kT = kHeadDim * kMergeSlices;
    __shared__ float wts[1024];
    __shared__ float red[kT / 32];
    __shared__ float so[kMergeSlices][kHeadDim];
    __shared__ float sl[kMergeSlices];
    pdl_wait();
    pdl_trigger();
    const int head = blockIdx.x, row = blockIdx.y, tid = threadIdx.x;
    const int d = tid & (kHeadDim - 1), slice = tid / kHeadDim;
    const int s = row_stream(a.rows, row);
    const int pos = a.rows.pos0[s] + (row - a.rows.row_start[s]);
    const int nb = pos / kKB + 1;
    const size_t base = ((size_t)row * a.n_q + head) * a.max_blocks;

    float M = -INFINITY;
    for (int b = tid; b < nb; b += kT) M = fmaxf(M, a.pm[base + b]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if ((tid & 31) == 0) red[tid >> 5] = M;
    __syncthreads();
    M = red[0];
#pragma unroll
    for (int w = 1; w < kT / 32; ++w) M = fmaxf(M, red[w]);

    float O = 0.f, L = 0.f;
    for (int c = 0; c < nb; c += 1024) {
        const int n = min(1024, nb - c);
        __syncthreads();
        for (int b = tid; b < n; b += kT) wts[b] = exp2f(a.pm[base + c + b] - M);
        __syncthreads();
        const float* pl = a.pl + base + c;
        const float* po = a.po + (base + c) * kHeadDim + d;
        int b = slice;
        for (; b + 7 * kMergeSlices < n; b += 8 * kMergeSlices) {
            float lv[8], ov[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                lv[u] = pl[b + u * kMergeSlices];
                ov[u] = po[(size_t)(b + u * kMergeSlices) * kHeadDim];
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                L = fmaf(lv[u], wts[b + u * kMergeSlices], L);
                O = fmaf(ov[u], wts[b + u * kMergeSlices], O);
            }
        }
        for (; b < n; b += kMergeSlices) {
            L = fmaf(pl[b], wts[b], L);
            O = fmaf(po[(size_t)b * kHeadDim], wts[b], O);
        }
    }
    so[slice][d] = O;
    if (d == 0) sl[slice] = L;
    __syncthreads();
    if (slice == 0) {
        O = so[0][d];
        L = sl[0];
#pragma unroll
        for (int i = 1; i < kMergeSlices; ++i) {
            O += so[i][d];
            L += sl[i];
        }
        a.out[(size_t)row * a.n_q * kHeadDim + (size_t)head * kHeadDim + d] = rn(O / L);
    }
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
    c2.blockDim = dim3(kHeadDim * kMergeSlices);
    c2.stream = st;
    c2.attrs = attr;
    c2.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&c2, attn_merge_kernel, a);
}

}  // namespace tfl
