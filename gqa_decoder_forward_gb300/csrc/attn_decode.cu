// Decode attention: causal GQA of a few rows per stream over a position-major
// paged bf16 cache, split over key units at absolute positions (pull request
// #1415, section "How": "decode rows on sdpa_vector lanes over key blocks at
// absolute positions").
//
// Pass 1 (attn_block_kernel): one CTA per (unit u of 512 positions, KV head g,
// group of <= 2 rows of one stream).  The unit's four 128-key sub-blocks of
// head g stream through two shared-memory buffers (cp.async), one computed
// while the next lands.  The G = n_q/n_kv query heads of the group's rows form
// the M dimension of tensor-core products (mma.sync m16n8k16, bf16 in, fp32
// accumulate); warp w owns keys 16w..16w+15 of every sub-block and runs its
// own online softmax (S = Q K^T, running max, O += P V), the warp partials are
// combined at the end.  Per (row, head) the CTA writes the unit's max score
// m_u, sum l_u = sum exp(s - m_u) and o_u = sum exp(s - m_u) v (attn_core.cuh).
// Pass 2 (attn_merge_kernel): per (row, head), M = max_u m_u, then
// L = sum_u l_u e^(m_u - M) and O = sum_u o_u e^(m_u - M) in unit order,
// out = bf16(O / L).
//
// Precision: scores are fp32 dot products of the bf16 q and k, scaled in fp32;
// softmax weights are fp32 and enter P V as a pair of bf16 numbers
// (hi = bf16(p), lo = bf16(p - hi)), i.e. with about 16 significant bits --
// the weights are not rounded to bf16.
//
// Determinism: every row's arithmetic depends only on its own position: the
// unit and sub-block split is fixed by absolute position, masked keys have
// weight exactly 0 (a sub-block past a row leaves its running values
// unchanged), keys past the last one any row of the group sees are zero-filled
// in shared memory, and each output element of an mma depends only on its own
// row of P.  A row gives the same bits alone or beside other rows (one-row
// steps == windows, solo == batched).
#include "common.cuh"
#include "attn_core.cuh"
#include "tma.cuh"
#include "warp_mma.cuh"

namespace tfl {
namespace {

constexpr int kThreads = 256;
constexpr int kRB = attn::kGroupRows;  // rows per CTA
constexpr int kSub = attn::kSub;
constexpr int kUnit = attn::kUnit;
using attn::swz;

// 202,304 bytes (one CTA per SM): queries, two buffers of one sub-block's
// keys and values each (sub-block j+1 streams in while j is computed), and the
// scratch that combines the eight warp partials.
struct Smem {
    bf16 q[attn::kPairs * kHeadDim];     // 4 KB
    bf16 k[2][kSub * kHeadDim];          // 2 x 32 KB
    bf16 v[2][kSub * kHeadDim];          // 2 x 32 KB
    float comb[attn::kCombFloats];       // 65 KB
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

// Sub-block staging through cp.async, two buffers (see attn::unit_partial for
// the contract): sub-block j lands in buffer j % 2 as one copy group; keys
// past the last visible one are zero-filled.
struct CpSrc {
    Smem* sm;
    const KvView* kv;
    int layer, n_kv, g, k0, p_last, nsub, issued;
    __device__ __forceinline__ void load(int j) {
        const int kj = k0 + j * kSub;
        const int nv = min(kSub, p_last + 1 - kj);
        const bf16* kbase = kv_row(*kv, layer, 0, kj, n_kv) + (size_t)g * kHeadDim;
        const bf16* vbase = kv_row(*kv, layer, 1, kj, n_kv) + (size_t)g * kHeadDim;
        const size_t pstride = (size_t)n_kv * kHeadDim;
        bf16* kd = sm->k[j & 1];
        bf16* vd = sm->v[j & 1];
        for (int i = threadIdx.x; i < kSub * 16; i += kThreads) {
            const int t = i >> 4, c = i & 15;
            const bool valid = t < nv;
            const size_t off = valid ? t * pstride + c * 8 : 0;
            cp_async16_zfill(kd + swz(t, c * 8), kbase + off, valid);
            cp_async16_zfill(vd + swz(t, c * 8), vbase + off, valid);
        }
        cp_async_commit();
        ++issued;
    }
    __device__ __forceinline__ uint32_t k(int j, int row, int col) const {
        return smem_u32(sm->k[j & 1]) + 2u * swz(row, col);
    }
    __device__ __forceinline__ uint32_t v(int j, int row, int col) const {
        return smem_u32(sm->v[j & 1]) + 2u * swz(row, col);
    }
    __device__ __forceinline__ void wait(int j) {
        if (issued > j + 1)
            cp_async_wait<1>();
        else
            cp_async_wait<0>();
        __syncthreads();
    }
    __device__ __forceinline__ void done(int j) {
        if (j + 2 < nsub) {
            __syncthreads();  // every warp is done with buffer j % 2
            load(j + 2);
        }
    }
};

// G = query heads per KV head.  Pair p = i*G + j is (row i of the group, head g*G + j).
template <int G>
__global__ void __launch_bounds__(kThreads, 1) attn_block_kernel(const __grid_constant__ AttnDecodeArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>(smem_raw);

    int s, r0, nr;
    if (!find_group(a.rows, blockIdx.z, s, r0, nr)) return;
    const int u = blockIdx.x, g = blockIdx.y;
    const int p_first = a.rows.pos0[s] + (r0 - a.rows.row_start[s]);
    const int p_last = p_first + nr - 1;
    const int k0 = u * kUnit;
    if (k0 > p_last) return;
    const int tid = threadIdx.x;
    const int P = nr * G;  // (row, head) pairs, at most 16

    CpSrc src;
    src.sm = &sm;
    src.kv = &a.rows.kv[s];
    src.layer = a.layer;
    src.n_kv = a.n_kv;
    src.g = g;
    src.k0 = k0;
    src.p_last = p_last;
    src.nsub = min(4, (p_last - k0) / kSub + 1);
    src.issued = 0;
    // A unit whose keys all precede the stream's first row of this call holds
    // cache rows written by earlier calls (every kernel of the library signals
    // its dependents only after its own dependency wait, so those writers have
    // completed): its first sub-blocks stream in while the previous kernel is
    // still finishing.
    const bool early = k0 + src.nsub * kSub <= a.rows.pos0[s];
    if (early) {
        src.load(0);
        if (src.nsub > 1) src.load(1);
    }
    pdl_wait();
    pdl_trigger();
    if (!early) {
        src.load(0);
        if (src.nsub > 1) src.load(1);
    }
    // queries (bf16, unscaled); pairs past P are zero
    for (int i = tid; i < attn::kPairs * 16; i += kThreads) {
        const int p = i >> 4, c = i & 15;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (p < P) {
            const int row = r0 + p / G, head = g * G + p % G;
            val = *reinterpret_cast<const uint4*>(a.q + (size_t)row * a.n_q * kHeadDim + (size_t)head * kHeadDim +
                                                   c * 8);
        }
        *reinterpret_cast<uint4*>(&sm.q[swz(p, c * 8)]) = val;
    }
    __syncthreads();  // the queries
    attn::UnitGeom ug;
    ug.u = u;
    ug.g = g;
    ug.r0 = r0;
    ug.P = P;
    ug.k0 = k0;
    ug.nsub = src.nsub;
    ug.p_first = p_first;
    ug.p_last = p_last;
    attn::unit_partial<G>(a, ug, smem_u32(sm.q), sm.comb, src, [] { __syncthreads(); });
}

// One CTA of 512 threads (a quarter of the units per 128) per (head, row).
__global__ void __launch_bounds__(512) attn_merge_kernel(const __grid_constant__ AttnDecodeArgs a) {
    __shared__ float red[512 / 32];
    __shared__ float2 part[attn::kQuarters * kHeadDim];
    pdl_wait();
    pdl_trigger();
    attn::merge<512>(a, blockIdx.y, blockIdx.x, threadIdx.x, red, part, [] { __syncthreads(); });
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
    return max_pos / kUnit + 1;
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
    c2.blockDim = dim3(512);
    c2.stream = st;
    c2.attrs = attr;
    c2.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&c2, attn_merge_kernel, a);
}

}  // namespace tfl
