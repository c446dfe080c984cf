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
#include "attn_core.cuh"
#include "tma.cuh"
#include "warp_mma.cuh"

namespace tfl {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = attn::kWarps;
constexpr int kRB = 4;               // rows per CTA
constexpr int kKB = attn::kKB;
constexpr int kMaxPairs = attn::kMaxPairs;
constexpr int kMergeSlices = attn::kMergeSlices;
using attn::swz;

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

    attn::BlockGeom bg;
    bg.b = b;
    bg.g = g;
    bg.r0 = r0;
    bg.P = P;
    bg.MT = MT;
    bg.k0 = k0;
    bg.nv = nv;
    bg.p_first = p_first;
    const uint32_t k_u = smem_u32(sm.k), v_u = smem_u32(sm.v);
    attn::block_partial<G>(
        a, bg, smem_u32(sm.q), k_u, sm.wmax, sm.wsum,
        [&](int row, int col) { return k_u + 2u * swz(row, col); },
        [&](int row, int col) { return v_u + 2u * swz(row, col); }, [] { __syncthreads(); },
        [] {
            cp_async_wait<0>();  // the values
            __syncthreads();
        });
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
    attn::merge<kT>(a, blockIdx.y, blockIdx.x, threadIdx.x, wts, red, so, sl, [] { __syncthreads(); });
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
