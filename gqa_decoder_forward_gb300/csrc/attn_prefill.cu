// Prompt-chunk attention: causal GQA of up to 2,048 rows of one stream over the
// paged cache (pull request #1415, section "How": prompt chunks attend the cache
// and the chunk's own earlier rows on the tensor units), one pass with an
// online softmax, the products on the 5th-generation tensor cores.
//
// One CTA per (query head h, pair of 128-row tiles A and B), 384 threads:
//   warps 0-3 softmax of tile A, warps 4-7 softmax of tile B: one thread per
//            query row (tensor-memory lane = row of the tile) holding the
//            row's 128 scores of a block in registers;
//   warp 8   TMA producer: both tiles' queries once, then the keys and values
//            of KV head h / G block by block (a block = 128 positions = one
//            cache page), double-buffered;
//   warps 10-11 idle (they complete the third warpgroup, whose registers the
//            softmax warpgroups take over);
//   warp 9   allocates tensor memory and issues the MMAs (one thread), per
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

constexpr int kThreads = 384;
// Registers: launched at 168 a thread (384 x 168 = 64,512); the producer/MMA
// warpgroup (warps 8-11) drops to kRegsLow, the two softmax warpgroups rise to
// kRegsHigh: 128 x 64 + 256 x 216 = 63,488 of the launch's 64,512.
constexpr int kRegsLow = 64, kRegsHigh = 216;
static_assert(128 * kRegsLow + 256 * kRegsHigh <= kThreads * 168, "register split exceeds the launch's registers");
constexpr int kBM = 128;                  // query rows per tile
constexpr int kBN = kPage;                // keys per block: one cache page
constexpr int kBox = 128 * 64 * 2;        // 16 KB: 128 rows x 64 columns, 128-byte swizzle
constexpr int kTile = 2 * kBox;           // 32 KB: 128 rows x 128 columns
constexpr int kTmemCols = 512;            // S/P of A, S/P of B, O of A, O of B: 128 columns each
constexpr float kScale = 0.12751743074640502f;  // log2(e) / sqrt(128)
constexpr float kRescale = 8.f;           // lazy rescale threshold (log2 units)

constexpr int kProducerWarp = 8, kMmaWarp = 9;

// Shared memory (from a 1024-byte aligned base): Q[2], K[2], V[2], barriers.
constexpr int kOffQ = 0, kOffK = 2 * kTile, kOffV = 4 * kTile;
constexpr int kOffBar = 6 * kTile;
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
            mbar_init(&b.p_full[i], kBM);
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

    if (warp >= 8) {
      // the third warpgroup: producer, MMA issuer, two idle warps
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
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
      }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsHigh));
        // ---------------- softmax: one thread per row ----------------
        // warps 4t .. 4t+3 serve tile t; warp w covers tensor-memory lanes
        // 32 (w mod 4) .. +31, i.e. rows of the tile, and holds a row's 128
        // scores of a block in registers (one load round trip, no exchange
        // with other threads)
        const int t = warp >> 2;
        const int row = (warp & 3) * 32 + lane;
        // this tile's geometry as scalars (a runtime index into the arrays would put them in local memory)
        const int t_r0 = t ? r0[1] : r0[0], t_nr = t ? nr[1] : nr[0], t_nb = t ? nbt[1] : nbt[0];
        const int pos = t ? min(p_first[1] + row, p_last[1]) : min(p_first[0] + row, p_last[0]);  // rows past the chunk see only real keys
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_off + t * 128, tO = tmem + lane_off + 256 + t * 128;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < t_nb; ++j) {
            if (ok && !*abort && !mbar_wait(&b.s_full[t], j & 1, a.status)) ok = false;
            tc_fence_after();
            const int k0 = j * kBN;
            const bool whole = k0 + kBN - 1 <= pos;  // every key of the block is visible to the row
            uint32_t sc[kBN];
            tmem_ld64_async(tS, sc);
            tmem_ld64_async(tS + 64, sc + 64);
            tmem_ld_wait();
            // keys past the row's position: score -inf, so that they take no part
            // in the max and get weight 2^-inf = 0 (only the blocks on the diagonal)
            if (!whole) {
#pragma unroll
                for (int e = 0; e < kBN; ++e)
                    if (k0 + e > pos) sc[e] = 0xFF800000u;
            }
            // block max (the scale is positive; a max is exact in any order)
            float mq[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) mq[e] = __uint_as_float(sc[e]);
#pragma unroll
            for (int e = 8; e < kBN; ++e) mq[e & 7] = fmaxf(mq[e & 7], __uint_as_float(sc[e]));
            const float bmax = fmaxf(fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])),
                                     fmaxf(fmaxf(mq[4], mq[5]), fmaxf(mq[6], mq[7]))) * kScale;
            const bool rescale = bmax > m + kRescale;  // a new reference max (always on block 0)
            const float alpha = rescale ? ex2(m - bmax) : 1.f;
            // O holds blocks 0 .. j-1 (this block's S was issued after that P V
            // finished); tensor-memory loads and stores take the whole warp, so
            // rows that keep their reference rewrite O times 1
            if (j > 0 && __any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
                for (int c = 0; c < kHeadDim / 16; ++c) {
                    float v[16];
                    tmem_ld16(tO + c * 16, v);
                    uint32_t w[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) w[e] = __float_as_uint(v[e] * alpha);
                    tmem_st16(tO + c * 16, w);
                }
            }
            if (rescale) {
                l *= alpha;
                m = bmax;
            }
            // weights p = 2^(s log2(e)/sqrt(128) - m), split into hi = bf16(p) and
            // lo = bf16(p - hi) (both rounded to nearest, unbiased), written over
            // the scores: for keys 32c .. 32c+31, hi in columns 32c .. 32c+15 and lo
            // in 32c+16 .. 32c+31; four running sums over keys 4i+0..3, added in
            // order at the end of the block
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c) {
                uint32_t w[32];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const int k = 32 * c + e;
                    const float p0 = ex2(fmaf(__uint_as_float(sc[k]), kScale, -m));
                    const float p1 = ex2(fmaf(__uint_as_float(sc[k + 1]), kScale, -m));
                    ls[e & 3] += p0;
                    ls[(e + 1) & 3] += p1;
                    const __nv_bfloat162 hh = __floats2bfloat162_rn(p0, p1);
                    w[e / 2] = *reinterpret_cast<const uint32_t*>(&hh);
                    w[16 + e / 2] = pack_rn(p0 - __low2float(hh), p1 - __high2float(hh));
                }
                tmem_st32(tS + c * 32, w);
            }
            l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            // values past the CTA's last position: exact zeros (the cache there holds anything)
            if (j == nb - 1 && k0 + row > p_end) {
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
        // the tile's last P V, then out = bf16(O / l)
        if (t_nb > 0) {
            if (ok && !*abort && !mbar_wait(&b.o_full[t], (t_nb - 1) & 1, a.status)) ok = false;
            tc_fence_after();
        }
        pdl_trigger();
        if (!ok) *abort = 1;
        if (t_nb > 0) {  // every lane loads (whole-warp instruction); rows of the chunk store
            bf16* out = a.out + (size_t)(t_r0 + row) * a.n_q * kHeadDim + (size_t)h * kHeadDim;
#pragma unroll 1
            for (int c = 0; c < kHeadDim / 32; ++c) {
                float v[32];
                tmem_ld32(tO + c * 32, v);
                if (row < t_nr) {
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
