// Prompt-chunk attention: causal GQA of up to 2,048 rows of one stream over the
// paged cache (pull request #1415, section "How": prompt chunks attend the cache
// and the chunk's own earlier rows on the tensor units), one pass with an
// online softmax, the products on the 5th-generation tensor cores.
//
// One CTA per (query head h, pair of 128-row tiles A and B), 576 threads:
//   warps 0-7 softmax of tile A, warps 8-15 softmax of tile B: two threads per
//            query row (tensor-memory lane = row of the tile), each over half
//            the keys of a block and half the output dims, the row max and
//            sum exchanged through shared memory;
//   warp 16  TMA producer: both tiles' queries once, then the keys and values
//            of KV head h / G block by block (a block = 128 positions = one
//            cache page), double-buffered;
//   warp 17  allocates tensor memory and issues the MMAs (one thread), per
//            block and tile: S = Q K^T (M = 128 rows, N = 128 keys, fp32 in
//            tensor memory), then O += P V (M = 128 rows, N = 128 dims) with the
//            weights P read from tensor memory, where the softmax wrote them
//            over S, and V read MN-major from shared memory.
// Tile B runs half a period behind tile A, so that while one tile's rows run
// their softmax the tensor cores work on the other tile; both tiles share each
// key/value block.
//
// Softmax of a row over block j: scores s (fp32 dot products of the bf16 q and
// k), visible keys only (causal), block max b = max(s) log2(e)/sqrt(128).  The
// row keeps a reference max m; when b > m + 8 (always on the first block) the
// reference becomes b and the running sum l and the tensor-memory output O are
// multiplied by 2^(m_old - m_new) (exactly the online softmax, rescaled lazily:
// every weight stays <= 2^8).  Weights p = 2^(s log2(e)/sqrt(128) - m) enter
// P V as hi = bf16(p) and lo = bf16(p - hi), both rounded to nearest (about
// 16 significant bits, unbiased; they are not rounded to bf16); l += sum p in
// a fixed order.  At the end out = bf16(O / l), rounded once.
//
// Determinism: a row's arithmetic depends only on the row and its position.
// Key blocks sit at absolute positions and are visited in order from 0; keys
// past a row's position have weight exactly 0 (a block past the row adds
// nothing and rescales nothing); values past the CTA's last position are
// zeroed in shared memory; every product element depends only on its own row
// of Q or P.  Chunk boundaries and a row's tile change no bits (a prompt
// resumed from a kept prefix equals the same prompt prefilled fresh).
#include "common.cuh"
#include "tcgen05.cuh"
#include "tma.cuh"

namespace tfl {
namespace {

constexpr int kThreads = 576;
constexpr int kBM = 128;                  // query rows per tile
constexpr int kBN = kPage;                // keys per block: one cache page
constexpr int kBox = 128 * 64 * 2;        // 16 KB: 128 rows x 64 columns, 128-byte swizzle
constexpr int kTile = 2 * kBox;           // 32 KB: 128 rows x 128 columns
constexpr int kTmemCols = 512;            // S/P of A, S/P of B, O of A, O of B: 128 columns each
constexpr float kScale = 0.12751743074640502f;  // log2(e) / sqrt(128)
constexpr float kRescale = 8.f;           // lazy rescale threshold (log2 units)

constexpr int kProducerWarp = 16, kMmaWarp = 17;

// Shared memory (from a 1024-byte aligned base): Q[2], K[2], V[2], the row-max
// exchange ([tile][block parity][half][row]) and row-sum exchange ([tile][half][row]), barriers.
constexpr int kOffQ = 0, kOffK = 2 * kTile, kOffV = 4 * kTile;
constexpr int kOffX = 6 * kTile;
constexpr int kOffBar = kOffX + (2 * 2 * 2 * 128 + 2 * 2 * 128) * 4;
constexpr int kSmem = 1024 + kOffBar + 16 * 8;

struct Bars {
    uint64_t q_full, kv_full[2], kv_empty[2], s_full[2], p_full[2], o_full[2];
    uint64_t drain;  // MMA completion after an abort
    uint32_t tmem;
    int abort;
};
static_assert(sizeof(Bars) <= 16 * 8, "barrier area");

// 2^x by the special-function unit (approximate, flushes subnormal results to
// zero; 2^-inf = 0).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_rn(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

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
    const int pair = gridDim.y - 1 - blockIdx.y;  // the longest tiles start first
    const int G = a.n_q / a.n_kv, g = h / G;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // tiles A (t = 0) and B (t = 1): rows, positions, key blocks
    int r0[2], nr[2], nbt[2], p_first[2], p_last[2];
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        r0[t] = (2 * pair + t) * kBM;
        nr[t] = min(kBM, a.n_rows - r0[t]);
        p_first[t] = a.pos0 + r0[t];
        p_last[t] = p_first[t] + nr[t] - 1;
        nbt[t] = nr[t] > 0 ? p_last[t] / kBN + 1 : 0;
    }
    const int nb = max(nbt[0], nbt[1]);
    const int p_end = nr[1] > 0 ? p_last[1] : p_last[0];  // the CTA's last position

    if (threadIdx.x == 0) {
        mbar_init(&b.q_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&b.kv_full[i], 1);
            mbar_init(&b.kv_empty[i], 1);
            mbar_init(&b.s_full[i], 1);
            mbar_init(&b.p_full[i], 2 * kBM);
            mbar_init(&b.o_full[i], 1);
        }
        mbar_init(&b.drain, 1);
        b.abort = 0;
        mbar_init_fence();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&b.tmem, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = b.tmem;
    bool mma_any = false;  // the MMA thread issued at least one MMA
    pdl_wait();

    if (warp == kProducerWarp) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            const uint64_t keep = policy_evict_last(), once = policy_evict_first();
            mbar_arrive_expect_tx(&b.q_full, 2 * kTile);
#pragma unroll
            for (int t = 0; t < 2; ++t) {  // rows past the chunk read as zeros
                tma_load_2d(base + kOffQ + t * kTile, &a.qmap, h * kHeadDim, r0[t], &b.q_full, once);
                tma_load_2d(base + kOffQ + t * kTile + kBox, &a.qmap, h * kHeadDim + 64, r0[t], &b.q_full, once);
            }
            int issued = 0;  // key/value blocks whose copies were issued
            for (int j = 0; j < nb && !*abort; ++j) {
                const int buf = j & 1;
                if (j >= 2 && !mbar_wait(&b.kv_empty[buf], ((j >> 1) - 1) & 1, a.status)) {
                    *abort = 1;
                    break;
                }
                issued = j + 1;
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
            // after an abort, the copies already issued land before the CTA exits
            // (blocks before the last two were released by the MMAs, so have landed)
            if (*abort) {
                mbar_wait(&b.q_full, 0u, a.status);
                for (int j = issued >= 2 ? issued - 2 : 0; j < issued; ++j)
                    mbar_wait(&b.kv_full[j & 1], (j >> 1) & 1, a.status);
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16_f32(kBM, kBN);
            constexpr uint32_t idPV = idesc_bf16_f32_bmn(kBM, kHeadDim);
            // S_t(j) into tile t's score columns (only after P V of block j-1,
            // which read the weights there, has finished)
            auto issue_s = [&](int t, int j) {
                tc_fence_after();
                const uint32_t kt = su + kOffK + (j & 1) * kTile;
#pragma unroll
                for (int kk = 0; kk < kHeadDim / 16; ++kk)
                    tc_mma_bf16(tmem + t * 128, kdesc(su + kOffQ + t * kTile, kk), kdesc(kt, kk), idS,
                                kk > 0 ? 1u : 0u);
                tc_commit(&b.s_full[t]);
            };
            // O_t += P_hi V + P_lo V of block j
            auto issue_pv = [&](int t, int j) {
                tc_fence_after();
                const uint32_t vt = su + kOffV + (j & 1) * kTile;
                const uint32_t tp = tmem + t * 128, to = tmem + 256 + t * 128;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    tc_mma_bf16_ta(to, tp + 32 * (kk >> 1) + 8 * (kk & 1), sdesc_sw128_mn(vt + kk * 2048, kBox), idPV,
                                   (j > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk)
                    tc_mma_bf16_ta(to, tp + 32 * (kk >> 1) + 16 + 8 * (kk & 1), sdesc_sw128_mn(vt + kk * 2048, kBox),
                                   idPV, 1u);
                tc_commit(&b.o_full[t]);
            };
            auto kv_ready = [&](int j) { return mbar_wait(&b.kv_full[j & 1], (j >> 1) & 1, a.status); };
            // Tile B runs half a period behind tile A: its first scores are issued
            // once A's first softmax is done, and from then on each tile's P V and
            // next S fill the tensor cores while the other tile's rows run their
            // softmax.
            bool ok = mbar_wait(&b.q_full, 0, a.status) && kv_ready(0);
            if (ok) issue_s(0, 0);
            mma_any = ok;
            for (int j = 0; j < nb && ok; ++j) {
                if (j < nbt[0]) {
                    if (!(ok = mbar_wait(&b.p_full[0], j & 1, a.status))) break;
                    if (j == 0 && nbt[1] > 0) issue_s(1, 0);
                    issue_pv(0, j);
                    if (j + 1 < nbt[0]) {
                        if (!(ok = mbar_wait(&b.o_full[0], j & 1, a.status) && kv_ready(j + 1))) break;
                        issue_s(0, j + 1);
                    }
                }
                if (j < nbt[1]) {
                    if (!(ok = mbar_wait(&b.p_full[1], j & 1, a.status))) break;
                    issue_pv(1, j);
                }
                tc_commit(&b.kv_empty[j & 1]);  // both tiles are done with block j
                if (j + 1 < nbt[1]) {
                    if (!(ok = mbar_wait(&b.o_full[1], j & 1, a.status) && kv_ready(j + 1))) break;
                    issue_s(1, j + 1);
                }
            }
            if (!ok) *abort = 1;
        }
    } else {
        // ---------------- softmax: two threads per row ----------------
        // warps 8t .. 8t+7 serve tile t; warp w covers tensor-memory lanes
        // 32 (w mod 4) .. +31 (the rows) and half (w / 4) mod 2 of the columns
        // (keys 64 hf .. 64 hf + 63 of S, dims 64 hf .. of O)
        const int t = warp >> 3, hf = (warp >> 2) & 1;
        const int row = (warp & 3) * 32 + lane;
        const int pos = min(p_first[t] + row, p_last[t]);  // rows past the chunk see only real keys
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_off + t * 128, tO = tmem + lane_off + 256 + t * 128 + hf * 64;
        float* xm = reinterpret_cast<float*>(base + kOffX) + t * (2 * 2 * kBM);  // [block parity][half][row]
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nbt[t]; ++j) {
            if (ok && !*abort && !mbar_wait(&b.s_full[t], j & 1, a.status)) ok = false;
            tc_fence_after();
            const int k0 = j * kBN, kh = k0 + hf * 64;  // first key of this thread's half
            const bool whole = k0 + kBN - 1 <= pos;      // every key of the block is visible to the row
            // pass 1: max of the visible raw scores of this half, then of the row
            float mx = -INFINITY;
            {
                float v[64];
                tmem_ld64(tS + hf * 64, v);
                if (whole) {
#pragma unroll
                    for (int e = 0; e < 64; ++e) mx = fmaxf(mx, v[e]);
                } else {
#pragma unroll
                    for (int e = 0; e < 64; ++e)
                        if (kh + e <= pos) mx = fmaxf(mx, v[e]);
                }
            }
            float* xj = xm + (j & 1) * (2 * kBM);
            xj[hf * kBM + row] = mx;
            named_barrier(1 + t, 8 * 32);
            mx = fmaxf(xj[row], xj[kBM + row]);
            const float bmax = mx * kScale;
            const bool rescale = bmax > m + kRescale;  // a new reference max (always on block 0)
            const float alpha = rescale ? ex2(m - bmax) : 1.f;
            // O holds blocks 0 .. j-1 (this block's S was issued after that P V
            // finished); tensor-memory loads and stores take the whole warp, so
            // rows that keep their reference rewrite O times 1
            if (j > 0 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    float v[32];
                    tmem_ld32(tO + c * 32, v);
                    uint32_t w[16];
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) w[e] = __float_as_uint(v[half * 16 + e] * alpha);
                        tmem_st16(tO + c * 32 + half * 16, w);
                    }
                }
            }
            if (rescale) {
                l *= alpha;
                m = bmax;
            }
            // pass 2: this half's weights (hi, lo) written over its scores; four
            // running sums over keys 4i+0..3, added in order at the end
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int c = 2 * hf + h2;  // keys 32c .. 32c+31 of the block
                float v[32];
                tmem_ld32(tS + c * 32, v);
                uint32_t hi[16], lo[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    float p0 = ex2(fmaf(v[e], kScale, -m));
                    float p1 = ex2(fmaf(v[e + 1], kScale, -m));
                    if (!whole) {
                        if (k0 + c * 32 + e > pos) p0 = 0.f;
                        if (k0 + c * 32 + e + 1 > pos) p1 = 0.f;
                    }
                    ls[e & 3] += p0;
                    ls[(e + 1) & 3] += p1;
                    // hi = bf16(p), lo = bf16(p - hi), both rounded to nearest (unbiased)
                    const __nv_bfloat162 hh = __floats2bfloat162_rn(p0, p1);
                    hi[e / 2] = *reinterpret_cast<const uint32_t*>(&hh);
                    lo[e / 2] = pack_rn(p0 - __low2float(hh), p1 - __high2float(hh));
                }
                // hi in columns 32c .. 32c+15, lo in 32c+16 .. 32c+31
                tmem_st16(tS + c * 32, hi);
                tmem_st16(tS + c * 32 + 16, lo);
            }
            l += (ls[0] + ls[1]) + (ls[2] + ls[3]);  // this half's running sum
            // values past the CTA's last position: exact zeros (the cache there holds anything)
            if (hf == 0 && j == nb - 1 && k0 + row > p_end) {
                const uint32_t vrow = su + kOffV + (j & 1) * kTile + row * 128;
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(vrow + ch * 16), "r"(0u) : "memory");
                    asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(vrow + kBox + ch * 16), "r"(0u)
                                 : "memory");
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&b.p_full[t]);
        }
        // the row's sum = first half's + second half's
        float* xl = reinterpret_cast<float*>(base + kOffX) + 2 * (2 * 2 * kBM) + t * (2 * kBM);
        xl[hf * kBM + row] = l;
        named_barrier(1 + t, 8 * 32);
        l = xl[row] + xl[kBM + row];
        // the tile's last P V, then out = bf16(O / l) for this half's 64 dims
        if (nbt[t] > 0) {
            if (ok && !*abort && !mbar_wait(&b.o_full[t], (nbt[t] - 1) & 1, a.status)) ok = false;
            tc_fence_after();
        }
        pdl_trigger();
        if (!ok) *abort = 1;
        if (nbt[t] > 0) {  // every lane loads (whole-warp instruction); rows of the chunk store
            bf16* out = a.out + (size_t)(r0[t] + row) * a.n_q * kHeadDim + (size_t)h * kHeadDim + hf * 64;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                float v[32];
                tmem_ld32(tO + c * 32, v);
                if (row < nr[t]) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 w;
                        w.x = pack_rn(v[8 * q + 0] / l, v[8 * q + 1] / l);
                        w.y = pack_rn(v[8 * q + 2] / l, v[8 * q + 3] / l);
                        w.z = pack_rn(v[8 * q + 4] / l, v[8 * q + 5] / l);
                        w.w = pack_rn(v[8 * q + 6] / l, v[8 * q + 7] / l);
                        *reinterpret_cast<uint4*>(out + c * 32 + 8 * q) = w;
                    }
                }
            }
        }
    }

    // every MMA was waited for by the softmax warps (or, after an abort, is waited
    // for below): free TMEM
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        // after an abort, every MMA already issued completes before tensor
        // memory is freed (a commit tracks all of this thread's earlier MMAs)
        if (lane == 0 && *abort && mma_any) {
            tc_commit(&b.drain);
            mbar_wait(&b.drain, 0u, a.status);
        }
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
    c.gridDim = dim3(a.n_q, (a.n_rows + 2 * kBM - 1) / (2 * kBM));
    c.blockDim = dim3(kThreads);
    c.dynamicSmemBytes = kSmem;
    c.stream = st;
    c.attrs = attr;
    c.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&c, attn_prefill_kernel, a);
}

}  // namespace tfl
