// Decode-row projections fed by TMA: y[r][n] = sum_k W[n][k] x[r][k] for 1..64
// activation rows, fp32 sums rounded once to bf16, with the op that follows
// the projection fused into the epilogue (row projections of pull request
// #1415, section "How": "decode windows on ll_matvec with fp32 sums rounded
// once").  The multiply is mma.sync m16n8k16 (bf16 in, fp32 accumulate).
//
// HBM-bound design: one persistent CTA per SM.  A producer warp streams stages
// of 16 weight rows x 512 columns (16 KB) with a single 3-D TMA load each
// (k-block as the outer box dimension, 128-byte swizzle) plus the matching
// 512 columns of the activation rows, into a ring of shared-memory stages
// (128 KB of weights in flight per SM for up to 8 rows).  Eight consumer
// warps each take one 64-column k-block of every stage, read their mma
// fragments from the swizzled tiles and release the stage through an
// mbarrier.  A work unit is one tile of 16 weight rows over the whole K, so
// every weight row is read as one contiguous stream; the 33B projections have
// 448 to 10,432 units, several per CTA.
//
// Determinism: warp w accumulates k-blocks w, w+8, w+16, ... of its tile in
// order; the eight warp sums are added in warp order.  Nothing depends on the
// number of activation rows, so a row's result is bit-identical alone or in a
// window of up to 64 rows.
//
// Tile rows (see matvec_epilogue.cuh): the 16 rows are 8 "lo" and 8 "hi" rows
//   STORE / RESIDUAL  rows 16t..16t+7 and 16t+8..16t+15
//   SWIGLU            gate rows 8t.. and up rows 8t.. (g and u of a feature)
//   QKV_ROPE          head h dims j0..j0+7 and j0+64.. (a NeoX RoPE pair)
#include <cuda.h>

#include "common.cuh"
#include "matvec_epilogue.cuh"
#include "rmsnorm_row.cuh"
#include "tma.cuh"

namespace tfl {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kKbPerStage = 8;                 // 8 x 64 columns per stage
constexpr int kABytes = 16 * 64 * 2 * kKbPerStage;  // 16 rows x 512 bf16 = 16 KB

// Shared memory of one CTA: a ring of `depth` stages (16 KB of weights plus
// the stage's activation rows, 1 KB per row) of up to 200 KB, the cross-warp
// sums and the barriers; the fused-norm variant keeps its normalised rows
// instead of per-stage activations.  (Rings of 128 KB and more stream at the
// same rate; 104 KB loses about 3% at one row.)
constexpr int kRing = 200 * 1024;
constexpr int kRedBytes(int nt) { return kConsumerWarps * nt * 4 * 32 * 4; }
constexpr int kRedNorm = 8 * 8 * 4;

int ring_depth(int stage_bytes, int budget) {
    int d = budget / stage_bytes;
    return d < 2 ? 2 : d > 8 ? 8 : d;
}
int stage_bytes_of(int x_rows_box, bool norm) { return kABytes + (norm ? 0 : x_rows_box * 1024); }
int smem_bytes(int nt, bool norm, int depth, int stage_bytes, int xn_bytes) {
    return 1024 + depth * stage_bytes + xn_bytes + kRedBytes(nt) + (norm ? kRedNorm : 0) + 2 * depth * 8 + 64;
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(addr));
    return r;
}

// The two 16-byte chunks (tig and tig+4) of 128-byte line `line` of a tile
// written by TMA with 128-byte swizzling (chunk c of line l sits at chunk
// c ^ (l mod 8)).  Lines with odd (l mod 8) read the upper chunk first, so each
// 8-lane phase of a warp touches 8 distinct bank groups.
__device__ __forceinline__ void line_chunks(uint32_t tile, int line, int tig, uint4& c0, uint4& c1) {
    const int sw = line & 7, odd = line & 1;
    const uint32_t row = tile + line * 128;
    uint4 a = lds128(row + (((tig + 4 * odd) ^ sw) << 4));
    uint4 b = lds128(row + (((tig + 4 * (1 - odd)) ^ sw) << 4));
    c0 = odd ? b : a;
    c1 = odd ? a : b;
}

__device__ __forceinline__ mv::TileRows tile_info(const MatvecArgs& e, int t) {
    mv::TileRows r;
    r.lo = r.hi = nullptr;
    r.seg = 0;
    r.head = 0;
    if (e.mode == MV_SWIGLU) {
        r.j0 = t * 8;
    } else if (e.mode == MV_QKV_ROPE) {
        const int tq = e.n_q * 8, tk = e.n_kv * 8;
        int u;
        if (t < tq) { r.seg = 0; u = t; }
        else if (t < tq + tk) { r.seg = 1; u = t - tq; }
        else { r.seg = 2; u = t - tq - tk; }
        r.head = u / 8;
        r.j0 = (u % 8) * 8;
    } else {
        r.j0 = t * 16;
    }
    return r;
}

// TMA loads of the 16 weight rows of tile t, k-blocks kb..kb+7, into sA:
// layout [k-block][16 rows][64], lo rows first.
__device__ __forceinline__ void load_weights(const MatvecTmaArgs& a, int t, int kb, unsigned char* sA,
                                             uint64_t* bar, uint64_t pol) {
    if (a.e.mode == MV_STORE || a.e.mode == MV_RESIDUAL) {
        tma_load_3d(sA, &a.wmap[0], 0, t * 16, kb, bar, pol);
    } else if (a.e.mode == MV_SWIGLU) {
        tma_load_3d(sA, &a.wmap[0], 0, t * 8, kb, bar, pol);          // gate rows (box of 8 rows)
        tma_load_3d(sA + kABytes / 2, &a.wmap[1], 0, t * 8, kb, bar, pol);  // up rows
    } else {
        const int tq = a.e.n_q * 8, tk = a.e.n_kv * 8;
        int seg, u;
        if (t < tq) { seg = 0; u = t; }
        else if (t < tq + tk) { seg = 1; u = t - tq; }
        else { seg = 2; u = t - tq - tk; }
        const int row = (u / 8) * kHeadDim + (u % 8) * 8;
        tma_load_3d(sA, &a.wmap[seg], 0, row, kb, bar, pol);
        tma_load_3d(sA + kABytes / 2, &a.wmap[seg], 0, row + 64, kb, bar, pol);
    }
}

// NORM: the activation rows are the residual stream a.e.x and are normalised
// (with a.norm_w) into shared memory by the consumers; requires NT == 1.
template <int NT, bool NORM>
__global__ void __launch_bounds__(kThreads, 1) matvec_tma_kernel(const __grid_constant__ MatvecTmaArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int depth = a.depth;
    const int stage_bytes = kABytes + (NORM ? 0 : a.x_rows_box * 1024);
    const int xn_bytes = NORM ? a.e.n_rows * a.e.K * 2 : 0;
    unsigned char* xn = base + depth * stage_bytes;  // NORM: [k-block][row][64], swizzled lines
    float* red = reinterpret_cast<float*>(xn + xn_bytes);
    float* red_norm = red + kConsumerWarps * NT * 4 * 32;
    uint64_t* full = reinterpret_cast<uint64_t*>(red_norm + (NORM ? 64 : 0));
    uint64_t* empty = full + depth;
    volatile int* s_abort = reinterpret_cast<volatile int*>(empty + depth);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tiles = a.tiles, nst = a.kstages;
    // stage bytes actually moved: weights (+ x rows present in the box)
    const uint32_t stage_tx = kABytes + (NORM ? 0 : a.x_rows_box * 128 * kKbPerStage);
    if (threadIdx.x == 0) {
        for (int s = 0; s < depth; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        *s_abort = 0;
        mbar_init_fence();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ---------------- producer ----------------
        if (lane == 0) {
            const uint64_t pw = policy_evict_first(), px = policy_evict_last();
            int t = blockIdx.x, ks = 0;
            // weight stages that fit the ring are issued before waiting for the
            // kernels that produce the activations
            int pre_ks[8];
            int n_pre = 0;
            while (n_pre < depth && t < tiles) {
                mbar_arrive_expect_tx(&full[n_pre], stage_tx);
                load_weights(a, t, ks * kKbPerStage, base + n_pre * stage_bytes, &full[n_pre], pw);
                pre_ks[n_pre++] = ks;
                if (++ks == nst) { ks = 0; t += gridDim.x; }
            }
            pdl_wait();
            pdl_trigger();
            if (!NORM)
                for (int i = 0; i < n_pre; ++i)
                    tma_load_3d(base + i * stage_bytes + kABytes, &a.xmap, 0, 0, pre_ks[i] * kKbPerStage, &full[i], px);
            int stage = n_pre % depth;
            uint32_t phase = n_pre == depth ? 1u : 0u;
            while (t < tiles) {
                if (*s_abort || !mbar_wait(&empty[stage], phase ^ 1u, a.status)) {
                    *s_abort = 1;
                    break;
                }
                unsigned char* sA = base + stage * stage_bytes;
                mbar_arrive_expect_tx(&full[stage], stage_tx);
                load_weights(a, t, ks * kKbPerStage, sA, &full[stage], pw);
                if (!NORM) tma_load_3d(sA + kABytes, &a.xmap, 0, 0, ks * kKbPerStage, &full[stage], px);
                if (++stage == depth) { stage = 0; phase ^= 1u; }
                if (++ks == nst) { ks = 0; t += gridDim.x; }
            }
            // after an abort, give copies already issued time to land before exiting
            if (*s_abort) __nanosleep(500000);
        } else {
            pdl_wait();
            pdl_trigger();
        }
        return;
    }

    // ---------------- consumers ----------------
    // the next kernel may launch once every CTA is past its dependency wait
    pdl_wait();
    pdl_trigger();
    const int g = lane >> 2, tig = lane & 3;
    const int R = a.e.n_rows, xrows = a.x_rows_box;
    const uint32_t base_u = smem_u32(base);
    const uint32_t xn_u = smem_u32(xn);
    const int kblocks = a.e.K / 64;
    if (NORM) {
        // the rows' RMSNorm, with the same arithmetic as the standalone norm kernel,
        // into [k-block][row][64] lines (chunk c of line l at c ^ (l mod 8))
        const int K = a.e.K, tid = threadIdx.x;
        for (int r = 0; r < R; ++r) {
            const bf16* hr = a.e.x + (size_t)r * K;
            const float rinv = rms_inv(hr, K, a.eps, tid, red_norm + r * 8, [] { named_barrier(1, kConsumerWarps * 32); });
            for (int i = tid * 8; i < K; i += kNormThreads * 8) {
                const uint4 hv = *reinterpret_cast<const uint4*>(hr + i);
                const uint4 wv = __ldg(reinterpret_cast<const uint4*>(a.norm_w + i));
                const bf16* he = reinterpret_cast<const bf16*>(&hv);
                const bf16* we = reinterpret_cast<const bf16*>(&wv);
                uint4 o;
                bf16* oe = reinterpret_cast<bf16*>(&o);
#pragma unroll
                for (int k = 0; k < 8; ++k) oe[k] = rms_apply(he[k], we[k], rinv);
                const int line = (i >> 6) * R + r, c = (i & 63) >> 3;
                asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(xn_u + line * 128 + ((c ^ (line & 7)) << 4)),
                             "r"(o.x), "r"(o.y), "r"(o.z), "r"(o.w)
                             : "memory");
            }
        }
        named_barrier(1, kConsumerWarps * 32);
    }
    // line of this warp's lo / hi weight row inside a stage: [k-block][16 rows]
    // for STORE/RESIDUAL; [k-block][8 lo rows] then [k-block][8 hi rows] otherwise
    const bool two_boxes = a.e.mode == MV_SWIGLU || a.e.mode == MV_QKV_ROPE;
    const int line_lo = two_boxes ? warp * 8 + g : warp * 16 + g;
    const int line_hi = two_boxes ? (kABytes / 2) / 128 + warp * 8 + g : warp * 16 + 8 + g;
    int stage = 0;
    uint32_t phase = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
        float acc[NT][4];
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
        for (int ks = 0; ks < nst; ++ks) {
            // after an abort every consumer keeps walking the loops (no more waits,
            // no early return) so that all of them reach the named barriers below
            if (!*s_abort && !mbar_wait(&full[stage], phase, a.status)) *s_abort = 1;
            const uint32_t sA = base_u + stage * stage_bytes;
            const uint32_t sX = sA + kABytes;
            const int kb = ks * kKbPerStage + warp;  // this warp's k-block
            uint4 l0, l1, h0, h1;
            line_chunks(sA, line_lo, tig, l0, l1);
            line_chunks(sA, line_hi, tig, h0, h1);
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const int xr = n * 8 + g;  // activation row of this lane's B fragment
                uint4 x0 = make_uint4(0u, 0u, 0u, 0u), x1 = x0;
                if (NORM) {
                    if (xr < R && kb < kblocks) line_chunks(xn_u, kb * R + xr, tig, x0, x1);
                } else if (xr < xrows) {
                    line_chunks(sX, warp * xrows + xr, tig, x0, x1);
                }
                mma16816(acc[n], l0.x, h0.x, l0.y, h0.y, x0.x, x0.y);
                mma16816(acc[n], l0.z, h0.z, l0.w, h0.w, x0.z, x0.w);
                mma16816(acc[n], l1.x, h1.x, l1.y, h1.y, x1.x, x1.y);
                mma16816(acc[n], l1.z, h1.z, l1.w, h1.w, x1.z, x1.w);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == depth) { stage = 0; phase ^= 1u; }
        }
        // fixed-order sum over the eight warps, then the epilogue
#pragma unroll
        for (int n = 0; n < NT; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i) red[((warp * NT + n) * 4 + i) * 32 + lane] = acc[n][i];
        named_barrier(1, kConsumerWarps * 32);
        const mv::TileRows tr = tile_info(a.e, t);
        for (int n = warp; n < NT; n += kConsumerWarps) {
            float v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float s = red[((0 * NT + n) * 4 + i) * 32 + lane];
#pragma unroll
                for (int w = 1; w < kConsumerWarps; ++w) s += red[((w * NT + n) * 4 + i) * 32 + lane];
                v[i] = s;
            }
            // c0 = (lo g, row 2tig), c1 = (lo g, row 2tig+1), c2 = (hi g, row 2tig), c3 = (hi g, row 2tig+1)
            const int r0 = n * 8 + 2 * tig;
            if (r0 < R) mv::epilogue(a.e, tr, g, r0, v[0], v[2]);
            if (r0 + 1 < R) mv::epilogue(a.e, tr, g, r0 + 1, v[1], v[3]);
        }
        named_barrier(1, kConsumerWarps * 32);
    }
}

template <int NT, bool NORM>
cudaError_t launch_nt(const MatvecTmaArgs& a, int grid, cudaStream_t st, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes =
        smem_bytes(NT, NORM, a.depth, stage_bytes_of(a.x_rows_box, NORM), NORM ? a.e.n_rows * a.e.K * 2 : 0);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, matvec_tma_kernel<NT, NORM>, a);
}

}  // namespace

int matvec_tma_nt(int n_rows) { return n_rows <= 8 ? 1 : n_rows <= 16 ? 2 : n_rows <= 32 ? 4 : 8; }

int matvec_tma_x_rows(int n_rows) { return n_rows <= 8 ? n_rows : 8 * matvec_tma_nt(n_rows); }

int matvec_tma_tiles(const MatvecArgs& e) {
    if (e.mode == MV_SWIGLU) return e.n_out / 8;
    if (e.mode == MV_QKV_ROPE) return (e.n_q + 2 * e.n_kv) * 8;
    return e.n_out / 16;
}

cudaError_t init_matvec_tma() {
    const int mx = 227 * 1024;
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(matvec_tma_kernel<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx)))
        return e;
    if ((e = cudaFuncSetAttribute(matvec_tma_kernel<2, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx)))
        return e;
    if ((e = cudaFuncSetAttribute(matvec_tma_kernel<4, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx)))
        return e;
    if ((e = cudaFuncSetAttribute(matvec_tma_kernel<8, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx)))
        return e;
    return cudaFuncSetAttribute(matvec_tma_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
}

// Ring depth of a launch (the fused-norm variant when norm is set).
int matvec_depth(int n_rows, int K, bool norm) {
    const int sb = stage_bytes_of(matvec_tma_x_rows(n_rows), norm);
    const int d = ring_depth(sb, kRing);
    if (norm) {
        // the normalised rows come on top of the ring: keep the CTA within 227 KB
        const int xn = n_rows * K * 2;
        int dd = d;
        while (dd > 2 && smem_bytes(1, true, dd, sb, xn) > 227 * 1024) --dd;
        return dd;
    }
    return d;
}

int matvec_norm_depth(int n_rows, int K) { return matvec_depth(n_rows, K, true); }

cudaError_t launch_matvec_tma(const MatvecTmaArgs& a0, int grid, cudaStream_t st, bool pdl) {
    MatvecTmaArgs a = a0;
    const int nt = matvec_tma_nt(a.e.n_rows);
    if (a.e.n_rows < 1 || a.e.n_rows > kMaxDecodeRows || a.kstages < 1 || a.tiles < 1 ||
        a.x_rows_box != matvec_tma_x_rows(a.e.n_rows) || a.e.K % 64 != 0 ||
        a.kstages != (a.e.K + 64 * kKbPerStage - 1) / (64 * kKbPerStage))
        return cudaErrorInvalidValue;
    if (grid > a.tiles) grid = a.tiles;
    const bool norm = a.norm_w != nullptr;
    a.depth = matvec_depth(a.e.n_rows, a.e.K, norm);
    const int sb = stage_bytes_of(a.x_rows_box, norm);
    if (smem_bytes(nt, norm, a.depth, sb, norm ? a.e.n_rows * a.e.K * 2 : 0) > 227 * 1024)
        return cudaErrorInvalidValue;
    if (norm) {
        if (nt != 1) return cudaErrorInvalidValue;
        return launch_nt<1, true>(a, grid, st, pdl);
    }
    switch (nt) {
        case 1: return launch_nt<1, false>(a, grid, st, pdl);
        case 2: return launch_nt<2, false>(a, grid, st, pdl);
        case 4: return launch_nt<4, false>(a, grid, st, pdl);
        default: return launch_nt<8, false>(a, grid, st, pdl);
    }
}

}  // namespace tfl
