// Prompt-chunk attention: causal GQA of up to 2,048 rows of one stream over the
// paged cache (pull request #1415, section "How": prompt chunks attend the cache
// and the chunk's own earlier rows), one pass with an online softmax.
//
// One CTA per (query head h, tile of 128 consecutive rows); 8 warps, 16 rows
// each.  The CTA walks the key blocks of 64 positions from position 0 up to the
// block of its last row, double-buffered in shared memory with cp.async (K and
// V of KV head h / G).  Per block and warp, on the tensor cores (mma.sync
// m16n8k16, bf16 in, fp32 accumulate): S = Q K^T for 16 rows x 64 keys, then
// the running row max m, rescale alpha = 2^(m_old - m_new) of the running sum l
// and of the output accumulator O, weights p = 2^(s - m_new), O += P V.
//
// Precision: scores are fp32 dot products of the bf16 q and k, scaled by
// log2(e)/sqrt(128) in fp32 so that exp2 gives e^(score/sqrt(128)); weights are
// fp32 and enter P V as a pair of bf16 numbers (hi = bf16(p), lo = bf16(p -
// hi)), about 16 significant bits -- they are not rounded to bf16.  The output
// is rounded to bf16 once, out = bf16(O / l).
//
// Determinism: a row's arithmetic depends only on the row and its position.
// Key blocks sit at absolute positions and are visited in order from 0; keys
// past a row's position have weight exactly 0 (so a block past the row is an
// exact no-op: alpha = 1, nothing added); keys past the tile's last row are
// zero-filled in shared memory; each mma output element depends only on its
// own row.  Chunk boundaries and a row's place in its tile change no bits
// (a prompt resumed from a kept prefix equals the same prompt prefilled fresh).
#include "common.cuh"
#include "warp_mma.cuh"

namespace tfl {
namespace {

using wm::cp_async16_zfill;
using wm::ldsm_x4;
using wm::ldsm_x4_t;
using wm::mma16816;
using wm::pack_bf16;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kBM = kWarps * 16;     // query rows per CTA
constexpr int kBN = 64;              // keys per block (divides the page of 128)
constexpr int kPad = kHeadDim + 8;   // padded row (bf16): 272 bytes, conflict-free ldmatrix

struct Smem {
    bf16 q[kBM][kPad];               // 34 KB
    bf16 k[2][kBN][kPad];            // 34 KB
    bf16 v[2][kBN][kPad];            // 34 KB
};

// Stages keys and values of KV head g for block j (positions 64j .. 64j+63, in
// one page); positions past p_last are zero-filled.
__device__ __forceinline__ void load_kv_block(Smem& sm, int buf, const AttnPrefillArgs& a, int g, int j, int p_last,
                                              int tid) {
    const int k0 = j * kBN;
    const bf16* kbase = kv_row(a.kv, a.layer, 0, k0, a.n_kv) + (size_t)g * kHeadDim;
    const bf16* vbase = kv_row(a.kv, a.layer, 1, k0, a.n_kv) + (size_t)g * kHeadDim;
    const size_t pstride = (size_t)a.n_kv * kHeadDim;
#pragma unroll
    for (int i = tid; i < kBN * 16; i += kThreads) {
        const int t = i >> 4, c = i & 15;
        const bool valid = k0 + t <= p_last;
        const size_t off = valid ? t * pstride + c * 8 : 0;
        cp_async16_zfill(&sm.k[buf][t][c * 8], kbase + off, valid);
        cp_async16_zfill(&sm.v[buf][t][c * 8], vbase + off, valid);
    }
    wm::cp_async_commit();
}

__global__ void __launch_bounds__(kThreads, 1) attn_prefill_kernel(const __grid_constant__ AttnPrefillArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
    const int h = blockIdx.x;
    const int tile = gridDim.y - 1 - blockIdx.y;  // the longest tiles start first
    const int G = a.n_q / a.n_kv, g = h / G;
    const int r0 = tile * kBM;
    const int nr = min(kBM, a.n_rows - r0);
    const int p_first = a.pos0 + r0;
    const int p_last = p_first + nr - 1;
    const int nb = p_last / kBN + 1;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, tig = lane & 3;
    const size_t ld = (size_t)a.n_q * kHeadDim;

    pdl_wait();
    load_kv_block(sm, 0, a, g, 0, p_last, tid);
    // queries of head h; rows past the chunk are zero
    for (int i = tid; i < kBM * 16; i += kThreads) {
        const int r = i >> 4, c = i & 15;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (r < nr) val = *reinterpret_cast<const uint4*>(a.q + (size_t)(r0 + r) * ld + (size_t)h * kHeadDim + c * 8);
        *reinterpret_cast<uint4*>(&sm.q[r][c * 8]) = val;
    }
    __syncthreads();
    uint32_t aq[kHeadDim / 16][4];
    {
        const int mrow = (lane & 7) + ((lane >> 3) & 1) * 8, mcol = (lane >> 4) * 8;
#pragma unroll
        for (int ks = 0; ks < kHeadDim / 16; ++ks) ldsm_x4(aq[ks], &sm.q[warp * 16 + mrow][ks * 16 + mcol]);
    }
    const int wr0 = warp * 16;
    const bool active = wr0 < nr;                           // warp holds chunk rows
    const int w_last = p_first + min(wr0 + 15, nr - 1);     // position of its last row
    const int pos_a = p_first + wr0 + gq, pos_b = pos_a + 8;  // this thread's two rows

    const float kScale = 0.12751743074640502f;  // log2(e) / sqrt(128)
    float o[kHeadDim / 8][4];
#pragma unroll
    for (int dt = 0; dt < kHeadDim / 8; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;
    const int krow = (lane & 7) + (lane >> 4) * 8, kcol = ((lane >> 3) & 1) * 8;
    const int vrow = (lane & 7) + ((lane >> 3) & 1) * 8, vcol = (lane >> 4) * 8;

    for (int j = 0; j < nb; ++j) {
        if (j + 1 < nb) {
            load_kv_block(sm, (j + 1) & 1, a, g, j + 1, p_last, tid);
            wm::cp_async_wait<1>();
        } else {
            wm::cp_async_wait<0>();
        }
        __syncthreads();
        const int buf = j & 1, k0 = j * kBN;
        if (active && k0 <= w_last) {
            // S = Q K^T over the block's 64 keys (8 n8 tiles)
            float s[kBN / 8][4];
#pragma unroll
            for (int nt = 0; nt < kBN / 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
            for (int ks = 0; ks < kHeadDim / 16; ++ks) {
#pragma unroll
                for (int np = 0; np < kBN / 16; ++np) {
                    uint32_t bk[4];
                    ldsm_x4(bk, &sm.k[buf][np * 16 + krow][ks * 16 + kcol]);
                    mma16816(s[2 * np], aq[ks], bk[0], bk[1]);
                    mma16816(s[2 * np + 1], aq[ks], bk[2], bk[3]);
                }
            }
            // scale, causal mask, block row maxima
            float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < kBN / 8; ++nt) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int t = k0 + nt * 8 + 2 * tig + e;
                    s[nt][e] = t <= pos_a ? s[nt][e] * kScale : -INFINITY;
                    s[nt][2 + e] = t <= pos_b ? s[nt][2 + e] * kScale : -INFINITY;
                    mx_a = fmaxf(mx_a, s[nt][e]);
                    mx_b = fmaxf(mx_b, s[nt][2 + e]);
                }
            }
            mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
            mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
            mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
            mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
            // key 0 is visible to every row, so the running max is finite after block 0
            const float mn_a = fmaxf(m_a, mx_a), mn_b = fmaxf(m_b, mx_b);
            const float al_a = exp2f(m_a - mn_a), al_b = exp2f(m_b - mn_b);
            m_a = mn_a;
            m_b = mn_b;
            // weights as hi/lo bf16 A fragments: k-step kk covers n8 tiles 2kk, 2kk+1
            uint32_t ph[kBN / 16][4], pl[kBN / 16][4];
            float sa = 0.f, sb = 0.f;
#pragma unroll
            for (int nt = 0; nt < kBN / 8; ++nt) {
                const float e0 = exp2f(s[nt][0] - mn_a), e1 = exp2f(s[nt][1] - mn_a);
                const float e2 = exp2f(s[nt][2] - mn_b), e3 = exp2f(s[nt][3] - mn_b);
                sa += e0;
                sa += e1;
                sb += e2;
                sb += e3;
                const bf16 h0 = rn(e0), h1 = rn(e1), h2 = rn(e2), h3 = rn(e3);
                const int kk = nt >> 1, half = nt & 1;
                ph[kk][half * 2 + 0] = pack_bf16(h0, h1);
                ph[kk][half * 2 + 1] = pack_bf16(h2, h3);
                pl[kk][half * 2 + 0] = pack_bf16(rn(e0 - bf(h0)), rn(e1 - bf(h1)));
                pl[kk][half * 2 + 1] = pack_bf16(rn(e2 - bf(h2)), rn(e3 - bf(h3)));
            }
            l_a = l_a * al_a + sa;
            l_b = l_b * al_b + sb;
#pragma unroll
            for (int dt = 0; dt < kHeadDim / 8; ++dt) {
                o[dt][0] *= al_a;
                o[dt][1] *= al_a;
                o[dt][2] *= al_b;
                o[dt][3] *= al_b;
            }
            // O += P V (hi part, then lo part)
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk) {
#pragma unroll
                for (int dp = 0; dp < kHeadDim / 16; ++dp) {
                    uint32_t bv[4];
                    ldsm_x4_t(bv, &sm.v[buf][kk * 16 + vrow][dp * 16 + vcol]);
                    mma16816(o[2 * dp], ph[kk], bv[0], bv[1]);
                    mma16816(o[2 * dp + 1], ph[kk], bv[2], bv[3]);
                    mma16816(o[2 * dp], pl[kk], bv[0], bv[1]);
                    mma16816(o[2 * dp + 1], pl[kk], bv[2], bv[3]);
                }
            }
        }
        __syncthreads();  // the buffer is refilled two blocks later
    }
    pdl_trigger();

    if (active) {
        float la = l_a + __shfl_xor_sync(0xffffffffu, l_a, 1);
        la += __shfl_xor_sync(0xffffffffu, la, 2);
        float lb = l_b + __shfl_xor_sync(0xffffffffu, l_b, 1);
        lb += __shfl_xor_sync(0xffffffffu, lb, 2);
        const int ra = wr0 + gq, rb = ra + 8;
        bf16* oa = a.out + (size_t)(r0 + ra) * ld + (size_t)h * kHeadDim + 2 * tig;
        bf16* ob = oa + 8 * ld;
#pragma unroll
        for (int dt = 0; dt < kHeadDim / 8; ++dt) {
            if (ra < nr)
                *reinterpret_cast<uint32_t*>(oa + dt * 8) = pack_bf16(rn(o[dt][0] / la), rn(o[dt][1] / la));
            if (rb < nr)
                *reinterpret_cast<uint32_t*>(ob + dt * 8) = pack_bf16(rn(o[dt][2] / lb), rn(o[dt][3] / lb));
        }
    }
}

}  // namespace

cudaError_t init_attn_prefill() {
    return cudaFuncSetAttribute(attn_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(Smem));
}

cudaError_t launch_attn_prefill(const AttnPrefillArgs& a, cudaStream_t st, bool pdl) {
    if (a.n_rows < 1 || a.n_kv < 1 || a.n_q < a.n_kv || a.n_q % a.n_kv != 0 || a.pos0 < 0)
        return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t c = {};
    c.gridDim = dim3(a.n_q, (a.n_rows + kBM - 1) / kBM);
    c.blockDim = dim3(kThreads);
    c.dynamicSmemBytes = (int)sizeof(Smem);
    c.stream = st;
    c.attrs = attr;
    c.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&c, attn_prefill_kernel, a);
}

}  // namespace tfl
