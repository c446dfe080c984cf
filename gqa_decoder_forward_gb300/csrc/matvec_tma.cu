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
#include "matvec_core.cuh"
#include "tma.cuh"

namespace tfl {
namespace {

using mvc::kABytes;
using mvc::kConsumerWarps;
using mvc::kKbPerStage;
constexpr int kThreads = (kConsumerWarps + 1) * 32;

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
            long long issued = 0;
            while (n_pre < depth && t < tiles) {
                mbar_arrive_expect_tx(&full[n_pre], stage_tx);
                mvc::load_weights(a.e, a.wmap, t, ks * kKbPerStage, base + n_pre * stage_bytes, &full[n_pre], pw);
                pre_ks[n_pre++] = ks;
                ++issued;
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
                mvc::load_weights(a.e, a.wmap, t, ks * kKbPerStage, sA, &full[stage], pw);
                if (!NORM) tma_load_3d(sA + kABytes, &a.xmap, 0, 0, ks * kKbPerStage, &full[stage], px);
                ++issued;
                if (++stage == depth) { stage = 0; phase ^= 1u; }
                if (++ks == nst) { ks = 0; t += gridDim.x; }
            }
            // after an abort, the copies already issued land before the CTA exits
            if (*s_abort) drain_ring(full, depth, stage, phase, issued, a.status);
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
    const int tig = lane & 3;
    const int R = a.e.n_rows, xrows = a.x_rows_box;
    const uint32_t base_u = smem_u32(base);
    const uint32_t xn_u = smem_u32(xn);
    const int kblocks = a.e.K / 64;
    const mvc::NamedBar1 bar;
    // NORM: the rows' RMSNorm, with the same arithmetic as the standalone norm
    // kernel, into [k-block][row][64] lines
    if (NORM)
        mvc::rows_to_lines([&](int r) { return a.e.x + (size_t)r * a.e.K; }, a.norm_w, a.eps, R, a.e.K, xn_u, red_norm,
                           bar);
    int stage = 0;
    uint32_t phase = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
        if (NORM)
            mvc::consume_tile<NT>(a.e, a.e.rows, t, nst, R, base_u, stage_bytes, depth, stage, phase, full, empty, red, s_abort,
                                  a.status, mvc::XFromLines{xn_u, R, kblocks, tig}, bar);
        else
            mvc::consume_tile<NT>(a.e, a.e.rows, t, nst, R, base_u, stage_bytes, depth, stage, phase, full, empty, red, s_abort,
                                  a.status, mvc::XFromStage{xrows, warp, tig}, bar);
    }
}

// Paired stages for 9 to 32 activation rows: a stage holds the weights of two
// adjacent tiles (2u and 2u+1) and one activation box, so each activation box
// streamed into shared memory serves 32 weight rows instead of 16 (at 16 rows
// the unpaired stage moves as many activation bytes as weight bytes).  Each
// tile's accumulation and cross-warp sum are those of matvec_tma_kernel, so
// the results are bit-identical to it.  Requires an even tile count.
__host__ __device__ constexpr int pair_stage_bytes(int x_rows_box) { return 2 * kABytes + x_rows_box * 1024; }

template <int NT>
__global__ void __launch_bounds__(kThreads, 1) matvec_tma_pair_kernel(const __grid_constant__ MatvecTmaArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int depth = a.depth;
    const int stage_bytes = pair_stage_bytes(a.x_rows_box);
    float* red = reinterpret_cast<float*>(base + depth * stage_bytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(red + kConsumerWarps * NT * 4 * 32);
    uint64_t* empty = full + depth;
    volatile int* s_abort = reinterpret_cast<volatile int*>(empty + depth);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int units = a.tiles / 2, nst = a.kstages;
    const uint32_t stage_tx = 2 * kABytes + a.x_rows_box * 128 * kKbPerStage;
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
            int u = blockIdx.x, ks = 0;
            auto weights = [&](unsigned char* sA, uint64_t* bar) {
                mvc::load_weights(a.e, a.wmap, 2 * u, ks * kKbPerStage, sA, bar, pw);
                mvc::load_weights(a.e, a.wmap, 2 * u + 1, ks * kKbPerStage, sA + kABytes, bar, pw);
            };
            // weight stages that fit the ring are issued before waiting for the
            // kernels that produce the activations
            int pre_ks[8];
            int n_pre = 0;
            long long issued = 0;
            while (n_pre < depth && u < units) {
                mbar_arrive_expect_tx(&full[n_pre], stage_tx);
                weights(base + n_pre * stage_bytes, &full[n_pre]);
                pre_ks[n_pre++] = ks;
                ++issued;
                if (++ks == nst) { ks = 0; u += gridDim.x; }
            }
            pdl_wait();
            pdl_trigger();
            for (int i = 0; i < n_pre; ++i)
                tma_load_3d(base + i * stage_bytes + 2 * kABytes, &a.xmap, 0, 0, pre_ks[i] * kKbPerStage, &full[i],
                            px);
            int stage = n_pre % depth;
            uint32_t phase = n_pre == depth ? 1u : 0u;
            while (u < units) {
                if (*s_abort || !mbar_wait(&empty[stage], phase ^ 1u, a.status)) {
                    *s_abort = 1;
                    break;
                }
                unsigned char* sA = base + stage * stage_bytes;
                mbar_arrive_expect_tx(&full[stage], stage_tx);
                weights(sA, &full[stage]);
                tma_load_3d(sA + 2 * kABytes, &a.xmap, 0, 0, ks * kKbPerStage, &full[stage], px);
                ++issued;
                if (++stage == depth) { stage = 0; phase ^= 1u; }
                if (++ks == nst) { ks = 0; u += gridDim.x; }
            }
            // after an abort, the copies already issued land before the CTA exits
            if (*s_abort) drain_ring(full, depth, stage, phase, issued, a.status);
        } else {
            pdl_wait();
            pdl_trigger();
        }
        return;
    }

    // ---------------- consumers ----------------
    pdl_wait();
    pdl_trigger();
    const int tig = lane & 3;
    const int R = a.e.n_rows, xrows = a.x_rows_box;
    const uint32_t base_u = smem_u32(base);
    const mvc::NamedBar1 bar;
    int stage = 0;
    uint32_t phase = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
        float acc[2][NT][4];
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int n = 0; n < NT; ++n) acc[t][n][0] = acc[t][n][1] = acc[t][n][2] = acc[t][n][3] = 0.f;
        mvc::accumulate_stages_pair<NT>(a.e, acc, 0, nst, base_u, stage_bytes, depth, stage, phase, full, empty,
                                        s_abort, a.status, mvc::XFromStage{xrows, warp, tig});
        mvc::finish_tile<NT>(a.e, a.e.rows, 2 * u, R, acc[0], red, bar);
        mvc::finish_tile<NT>(a.e, a.e.rows, 2 * u + 1, R, acc[1], red, bar);
    }
}

template <int NT>
cudaError_t launch_pair(const MatvecTmaArgs& a, int grid, cudaStream_t st, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes(NT, false, a.depth, pair_stage_bytes(a.x_rows_box), 0);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, matvec_tma_pair_kernel<NT>, a);
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
    if ((e = cudaFuncSetAttribute(matvec_tma_pair_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx)))
        return e;
    if ((e = cudaFuncSetAttribute(matvec_tma_pair_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx)))
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
    const bool norm = a.norm_w != nullptr;
    if (!norm && (nt == 2 || nt == 4) && a.tiles % 2 == 0) {
        // paired stages: each activation box serves two tiles
        const int sb = pair_stage_bytes(a.x_rows_box);
        a.depth = ring_depth(sb, kRing);
        if (smem_bytes(nt, false, a.depth, sb, 0) > 227 * 1024) return cudaErrorInvalidValue;
        if (grid > a.tiles / 2) grid = a.tiles / 2;
        return nt == 2 ? launch_pair<2>(a, grid, st, pdl) : launch_pair<4>(a, grid, st, pdl);
    }
    if (grid > a.tiles) grid = a.tiles;
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
