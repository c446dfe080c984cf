// Prompt-chunk attention: causal GQA of up to 2,048 rows of one stream over the
// paged cache (pull request #1415, section "How": prompt chunks attend the cache
// and the chunk's own earlier rows on the tensor units), one pass with an
// online softmax, the products on the 5th-generation tensor cores.
//
// One CTA per (query head h, tile of 128 consecutive rows), 192 threads:
//   warp 0   TMA producer: the tile's queries once, then the keys and values of
//            KV head h / G block by block (a block = 128 positions = one cache
//            page), double-buffered;
//   warp 1   allocates tensor memory and issues the MMAs (one thread):
//            S = Q K^T into tensor memory (M = 128 rows, N = 128 keys, fp32),
//            then O_blk = P_hi V + P_lo V (M = 128 rows, N = 128 dims) with the
//            weights P from shared memory and V read MN-major;
//   warps 2-5 one query row per thread (tensor-memory lane = row): read the
//            row of S, causal mask, block max, weights p = 2^(s - m_new) as a
//            pair of bf16 numbers into shared memory, running sum; then fold
//            the block's O_blk into the row's fp32 output in registers,
//            O = O 2^(m_old - m_new) + O_blk; at the end out = bf16(O / l).
// The next block's S = Q K^T is issued before this block's P V, and a row's
// max pass over the next block runs while P V is in flight.
//
// Precision: scores are fp32 dot products of the bf16 q and k, scaled by
// log2(e)/sqrt(128) in fp32 so that exp2 gives e^(score/sqrt(128)); weights are
// fp32 and enter P V as hi = bf16(p) and lo = bf16(p - hi) (about 16
// significant bits) -- they are not rounded to bf16.  The output is rounded
// to bf16 once.
//
// Determinism: a row's arithmetic depends only on the row and its position.
// Key blocks sit at absolute positions and are visited in order from 0; keys
// past a row's position have weight exactly 0 (a block past the row changes
// nothing: the max stays, the rescale factor is 1, O_blk of the row is 0);
// values past the tile's last position are zeroed in shared memory; every
// product element depends only on its own row of Q or P.  Chunk boundaries and
// a row's place in its tile change no bits (a prompt resumed from a kept prefix
// equals the same prompt prefilled fresh).
#include "common.cuh"
#include "tcgen05.cuh"
#include "tma.cuh"
#include "warp_mma.cuh"

namespace tfl {
namespace {

constexpr int kThreads = 192;
constexpr int kBM = 128;                  // query rows per CTA
constexpr int kBN = kPage;                // keys per block: one cache page
constexpr int kBox = 128 * 64 * 2;        // 16 KB: 128 rows x 64 columns, 128-byte swizzle
constexpr int kTile = 2 * kBox;           // 32 KB: 128 rows x 128 columns
constexpr int kTmemCols = 256;            // S: columns 0..127, O_blk: 128..255
constexpr float kScale = 0.12751743074640502f;  // log2(e) / sqrt(128)
using wm::pack_bf16;

// 2^x by the special-function unit (approximate, flushes subnormal results to
// zero; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Shared memory (from a 1024-byte aligned base): Q, K[2], V[2], P_hi, P_lo, barriers.
constexpr int kOffQ = 0, kOffK = kTile, kOffV = 3 * kTile, kOffPh = 5 * kTile, kOffPl = 6 * kTile;
constexpr int kOffBar = 7 * kTile;
constexpr int kSmem = 1024 + kOffBar + 16 * 8;

struct Bars {
    uint64_t q_full, kv_full[2], kv_empty[2], s_full, s_empty, p_full, o_full, o_empty;
    uint32_t tmem;
    int abort;
};

// Descriptor of the K-major 128 x 128 tile at `tile` (two 64-column boxes) for k-step kk (16 columns).
__device__ __forceinline__ uint64_t kdesc(uint32_t tile, int kk) {
    return sdesc_sw128(tile + (kk >> 2) * kBox + (kk & 3) * 32);
}

__global__ void __launch_bounds__(kThreads, 1) attn_prefill_kernel(const __grid_constant__ AttnPrefillArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars& b = *reinterpret_cast<Bars*>(base + kOffBar);
    volatile int* abort = &b.abort;
    const uint32_t su = smem_u32(base);
    const int h = blockIdx.x;
    const int tile = gridDim.y - 1 - blockIdx.y;  // the longest tiles start first
    const int G = a.n_q / a.n_kv, g = h / G;
    const int r0 = tile * kBM;
    const int nr = min(kBM, a.n_rows - r0);
    const int p_first = a.pos0 + r0;
    const int p_last = p_first + nr - 1;
    const int nb = p_last / kBN + 1;  // key blocks 0 .. nb-1
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(&b.q_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&b.kv_full[i], 1);
            mbar_init(&b.kv_empty[i], 1);
        }
        mbar_init(&b.s_full, 1);
        mbar_init(&b.s_empty, kBM);
        mbar_init(&b.p_full, kBM);
        mbar_init(&b.o_full, 1);
        mbar_init(&b.o_empty, kBM);
        b.abort = 0;
        mbar_init_fence();
    }
    if (warp == 1) {
        tmem_alloc(&b.tmem, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = b.tmem;
    pdl_wait();

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            const uint64_t keep = policy_evict_last(), once = policy_evict_first();
            mbar_arrive_expect_tx(&b.q_full, kTile);
            tma_load_2d(base + kOffQ, &a.qmap, h * kHeadDim, r0, &b.q_full, once);
            tma_load_2d(base + kOffQ + kBox, &a.qmap, h * kHeadDim + 64, r0, &b.q_full, once);
            for (int j = 0; j < nb && !*abort; ++j) {
                const int buf = j & 1;
                if (j >= 2 && !mbar_wait(&b.kv_empty[buf], ((j >> 1) - 1) & 1, a.status)) {
                    *abort = 1;
                    break;
                }
                const int page = __ldg(a.kv.table + j);
                mbar_arrive_expect_tx(&b.kv_full[buf], 2 * kTile);
#pragma unroll
                for (int kind = 0; kind < 2; ++kind) {
                    const int row0 = ((a.layer * 2 + kind) * a.kv.n_pages + page) * kPage;
                    unsigned char* dst = base + (kind ? kOffV : kOffK) + buf * kTile;
                    tma_load_3d(dst, &a.kvmap, 0, g, row0, &b.kv_full[buf], keep);
                    tma_load_3d(dst + kBox, &a.kvmap, 64, g, row0, &b.kv_full[buf], keep);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_f32(kBM, kBN);
            constexpr uint32_t idPV = idesc_bf16_f32_bmn(kBM, kHeadDim);
            const uint32_t tS = tmem, tO = tmem + 128;
            auto issue_s = [&](int j) -> bool {
                const int buf = j & 1;
                if (!mbar_wait(&b.kv_full[buf], (j >> 1) & 1, a.status)) return false;
                if (j > 0 && !mbar_wait(&b.s_empty, (j - 1) & 1, a.status)) return false;
                tc_fence_after();
                const uint32_t kt = su + kOffK + buf * kTile;
#pragma unroll
                for (int kk = 0; kk < kHeadDim / 16; ++kk)
                    tc_mma_bf16(tS, kdesc(su + kOffQ, kk), kdesc(kt, kk), idS, kk > 0 ? 1u : 0u);
                tc_commit(&b.s_full);
                return true;
            };
            bool ok = mbar_wait(&b.q_full, 0, a.status) && issue_s(0);
            for (int j = 0; j < nb && ok; ++j) {
                const int buf = j & 1;
                if (j + 1 < nb && !issue_s(j + 1)) {
                    ok = false;
                    break;
                }
                // O_blk = P_hi V + P_lo V once the weights are written and the
                // previous O_blk has been read
                if (!mbar_wait(&b.p_full, j & 1, a.status) || (j > 0 && !mbar_wait(&b.o_empty, (j - 1) & 1, a.status))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t vt = su + kOffV + buf * kTile;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    tc_mma_bf16(tO, kdesc(su + kOffPh, kk), sdesc_sw128_mn(vt + kk * 2048, kBox), idPV, kk > 0 ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    tc_mma_bf16(tO, kdesc(su + kOffPl, kk), sdesc_sw128_mn(vt + kk * 2048, kBox), idPV, 1u);
                tc_commit(&b.o_full);
                tc_commit(&b.kv_empty[buf]);
            }
            if (!ok) *abort = 1;
        }
    } else {
        // ---------------- softmax: one row per thread ----------------
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        const int pos = min(p_first + row, p_last);  // rows past the chunk see only real keys
        const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_off, tO = tmem + lane_off + 128;
        float o[kHeadDim];
#pragma unroll
        for (int d = 0; d < kHeadDim; ++d) o[d] = 0.f;
        float m = -INFINITY, l = 0.f, alpha_prev = 1.f;
        bool ok = true;
        // O += O_blk of block j, rescaled by alpha (the factor from block j-1's max to block j's)
        auto fold_o = [&](int j, float alpha) {
            if (ok && !*abort && !mbar_wait(&b.o_full, j & 1, a.status)) ok = false;
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < kHeadDim / 32; ++c) {
                float v[32];
                tmem_ld32(tO + c * 32, v);
#pragma unroll
                for (int e = 0; e < 32; ++e) o[c * 32 + e] = fmaf(o[c * 32 + e], alpha, v[e]);
            }
            tc_fence_before();
            mbar_arrive(&b.o_empty);
        };
        for (int j = 0; j < nb; ++j) {
            if (ok && !*abort && !mbar_wait(&b.s_full, j & 1, a.status)) ok = false;
            tc_fence_after();
            const int k0 = j * kBN;
            const bool whole = k0 + kBN - 1 <= pos;  // every key of the block is visible to the row
            // pass 1: block max of the visible raw scores (the scale is positive)
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c) {
                float v[32];
                tmem_ld32(tS + c * 32, v);
                if (whole) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) mx = fmaxf(mx, v[e]);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (k0 + c * 32 + e <= pos) mx = fmaxf(mx, v[e]);
                }
            }
            const float m_new = fmaxf(m, mx * kScale);
            const float alpha = ex2(m - m_new);
            // the previous block's O_blk (P V finished, so P may be rewritten)
            if (j > 0) fold_o(j - 1, alpha_prev);
            // pass 2: weights p = 2^(s scale - m_new) as (hi, lo) into shared
            // memory; four running sums over keys 4i+0..3, added in order at the end
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c) {
                float v[32];
                tmem_ld32(tS + c * 32, v);
                uint32_t hi[16], lo[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    float p0 = ex2(fmaf(v[e], kScale, -m_new)), p1 = ex2(fmaf(v[e + 1], kScale, -m_new));
                    if (!whole) {
                        if (k0 + c * 32 + e > pos) p0 = 0.f;
                        if (k0 + c * 32 + e + 1 > pos) p1 = 0.f;
                    }
                    ls[e & 3] += p0;
                    ls[(e + 1) & 3] += p1;
                    const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
                    const __nv_bfloat162 r = __floats2bfloat162_rn(p0 - __low2float(h), p1 - __high2float(h));
                    hi[e / 2] = *reinterpret_cast<const uint32_t*>(&h);
                    lo[e / 2] = *reinterpret_cast<const uint32_t*>(&r);
                }
                // keys 32c .. 32c+31 = chunks 4c .. 4c+3 of the row (box c / 2)
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const int ch = (4 * c + q4) & 7;
                    const uint32_t off = (c >> 1) * kBox + row * 128 + ((ch ^ (row & 7)) << 4);
                    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(su + kOffPh + off), "r"(hi[4 * q4]),
                                 "r"(hi[4 * q4 + 1]), "r"(hi[4 * q4 + 2]), "r"(hi[4 * q4 + 3])
                                 : "memory");
                    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(su + kOffPl + off), "r"(lo[4 * q4]),
                                 "r"(lo[4 * q4 + 1]), "r"(lo[4 * q4 + 2]), "r"(lo[4 * q4 + 3])
                                 : "memory");
                }
            }
            const float lsum = (ls[0] + ls[1]) + (ls[2] + ls[3]);
            tc_fence_before();
            mbar_arrive(&b.s_empty);
            // values past the tile's last position: exact zeros (the cache there holds anything)
            if (j == nb - 1 && k0 + row > p_last) {
                const uint32_t vrow = su + kOffV + (j & 1) * kTile + row * 128;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(vrow + ch * 16), "r"(0u) : "memory");
                    asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(vrow + kBox + ch * 16), "r"(0u)
                                 : "memory");
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive(&b.p_full);
            l = l * alpha + lsum;
            m = m_new;
            alpha_prev = alpha;
        }
        fold_o(nb - 1, alpha_prev);
        pdl_trigger();
        if (!ok) *abort = 1;
        if (row < nr) {
            bf16* out = a.out + (size_t)(r0 + row) * a.n_q * kHeadDim + (size_t)h * kHeadDim;
#pragma unroll
            for (int c = 0; c < kHeadDim / 8; ++c) {
                uint4 w;
                w.x = pack_bf16(rn(o[8 * c + 0] / l), rn(o[8 * c + 1] / l));
                w.y = pack_bf16(rn(o[8 * c + 2] / l), rn(o[8 * c + 3] / l));
                w.z = pack_bf16(rn(o[8 * c + 4] / l), rn(o[8 * c + 5] / l));
                w.w = pack_bf16(rn(o[8 * c + 6] / l), rn(o[8 * c + 7] / l));
                *reinterpret_cast<uint4*>(out + 8 * c) = w;
            }
        }
    }

    // every MMA was waited for by the softmax warps (or the kernel gave up): free TMEM
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        if (*abort) __nanosleep(500000);  // let copies and MMAs already issued finish
        tc_fence_after();
        __syncwarp();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t init_attn_prefill() {
    return cudaFuncSetAttribute(attn_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
}

cudaError_t launch_attn_prefill(const AttnPrefillArgs& a, cudaStream_t st, bool pdl) {
    if (a.n_rows < 1 || a.n_kv < 1 || a.n_q < a.n_kv || a.n_q % a.n_kv != 0 || a.pos0 < 0 ||
        (a.pos0 + a.n_rows - 1) / kPage >= a.kv.n_pages)
        return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t c = {};
    c.gridDim = dim3(a.n_q, (a.n_rows + kBM - 1) / kBM);
    c.blockDim = dim3(kThreads);
    c.dynamicSmemBytes = kSmem;
    c.stream = st;
    c.attrs = attr;
    c.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&c, attn_prefill_kernel, a);
}

}  // namespace tfl
