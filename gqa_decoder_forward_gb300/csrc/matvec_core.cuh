// The arithmetic of the decode matvec (y = W x for up to 64 activation rows),
// shared by the projection kernels and the persistent decode-step kernel so
// that both give the same bits: weight stages of 16 rows x 512 columns written
// by one 3-D TMA load (k-block outermost, 128-byte swizzle), fragments read with
// swizzle-aware 16-byte loads, mma.sync m16n8k16 (bf16 in, fp32 accumulate),
// warp w taking k-block w of every stage, a fixed-order sum over the eight
// warps, then the fused epilogue.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "matvec_epilogue.cuh"
#include "rmsnorm_row.cuh"
#include "tma.cuh"

namespace tfl {
namespace mvc {

constexpr int kConsumerWarps = 8;
constexpr int kKbPerStage = 8;                      // 8 x 64 columns per stage
constexpr int kABytes = 16 * 64 * 2 * kKbPerStage;  // 16 rows x 512 bf16 = 16 KB

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
__device__ __forceinline__ void load_weights(const MatvecArgs& e, const CUtensorMap* wmap, int t, int kb,
                                             unsigned char* sA, uint64_t* bar, uint64_t pol) {
    if (e.mode == MV_STORE || e.mode == MV_RESIDUAL) {
        tma_load_3d(sA, &wmap[0], 0, t * 16, kb, bar, pol);
    } else if (e.mode == MV_SWIGLU) {
        tma_load_3d(sA, &wmap[0], 0, t * 8, kb, bar, pol);          // gate rows (box of 8 rows)
        tma_load_3d(sA + kABytes / 2, &wmap[1], 0, t * 8, kb, bar, pol);  // up rows
    } else {
        const int tq = e.n_q * 8, tk = e.n_kv * 8;
        int seg, u;
        if (t < tq) { seg = 0; u = t; }
        else if (t < tq + tk) { seg = 1; u = t - tq; }
        else { seg = 2; u = t - tq - tk; }
        const int row = (u / 8) * kHeadDim + (u % 8) * 8;
        tma_load_3d(sA, &wmap[seg], 0, row, kb, bar, pol);
        tma_load_3d(sA + kABytes / 2, &wmap[seg], 0, row + 64, kb, bar, pol);
    }
}


// B-fragment sources for consume_tile: the activation tile of the stage (rows
// [warp][xrows][64] per k-block) or activation lines kept in shared memory.
struct XFromStage {
    int xrows, warp, tig;
    __device__ __forceinline__ void operator()(int xr, int, uint32_t sX, uint4& x0, uint4& x1) const {
        if (xr < xrows) line_chunks(sX, warp * xrows + xr, tig, x0, x1);
    }
};
struct XFromLines {
    uint32_t xs_u;
    int R, kblocks, tig;
    __device__ __forceinline__ void operator()(int xr, int kb, uint32_t, uint4& x0, uint4& x1) const {
        if (xr < R && kb < kblocks) line_chunks(xs_u, kb * R + xr, tig, x0, x1);
    }
};
struct NamedBar1 {
    __device__ __forceinline__ void operator()() const { named_barrier(1, kConsumerWarps * 32); }
};


// Accumulates stages ks0 .. ks1-1 of a tile into acc (consumer warps 0..7 of
// the CTA, ring of `depth` stages of stage_bytes at base_u): warp w takes
// k-block w of every stage.  xfrag(xr, kb, sX, x0, x1) fills the B fragment
// (16-byte chunks tig and tig+4 of k-block kb) of activation row xr (< 8 * NT),
// or leaves it zero.  After a failed wait the loop keeps walking (no more
// waits) so that every consumer reaches the barriers.
template <int NT, class XFrag>
__device__ __forceinline__ void accumulate_stages(const MatvecArgs& e, float (&acc)[NT][4], int ks0, int ks1,
                                                  uint32_t base_u, int stage_bytes, int depth, int& stage,
                                                  uint32_t& phase, uint64_t* full, uint64_t* empty,
                                                  volatile int* s_abort, int* status, XFrag xfrag) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tig = lane & 3;
    // line of this warp's lo / hi weight row inside a stage: [k-block][16 rows]
    // for STORE/RESIDUAL; [k-block][8 lo rows] then [k-block][8 hi rows] otherwise
    const bool two_boxes = e.mode == MV_SWIGLU || e.mode == MV_QKV_ROPE;
    const int line_lo = two_boxes ? warp * 8 + g : warp * 16 + g;
    const int line_hi = two_boxes ? (kABytes / 2) / 128 + warp * 8 + g : warp * 16 + 8 + g;
    for (int ks = ks0; ks < ks1; ++ks) {
        if (!*s_abort && !mbar_wait(&full[stage], phase, status)) *s_abort = 1;
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
            xfrag(xr, kb, sX, x0, x1);
            mma16816(acc[n], l0.x, h0.x, l0.y, h0.y, x0.x, x0.y);
            mma16816(acc[n], l0.z, h0.z, l0.w, h0.w, x0.z, x0.w);
            mma16816(acc[n], l1.x, h1.x, l1.y, h1.y, x1.x, x1.y);
            mma16816(acc[n], l1.z, h1.z, l1.w, h1.w, x1.z, x1.w);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
        if (++stage == depth) { stage = 0; phase ^= 1u; }
    }
}

// The same for a stage that holds two tiles' weights (tile A at sA, tile B at
// sA + kABytes) and one activation box after them (at sA + 2 kABytes): each
// warp reads its activation fragments once and runs the same mma sequence on
// both tiles, so every output element accumulates exactly as in
// accumulate_stages.  XFromStage-style fragments only (sX is passed).
template <int NT, class XFrag>
__device__ __forceinline__ void accumulate_stages_pair(const MatvecArgs& e, float (&acc)[2][NT][4], int ks0, int ks1,
                                                       uint32_t base_u, int stage_bytes, int depth, int& stage,
                                                       uint32_t& phase, uint64_t* full, uint64_t* empty,
                                                       volatile int* s_abort, int* status, XFrag xfrag) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tig = lane & 3;
    const bool two_boxes = e.mode == MV_SWIGLU || e.mode == MV_QKV_ROPE;
    const int line_lo = two_boxes ? warp * 8 + g : warp * 16 + g;
    const int line_hi = two_boxes ? (kABytes / 2) / 128 + warp * 8 + g : warp * 16 + 8 + g;
    for (int ks = ks0; ks < ks1; ++ks) {
        if (!*s_abort && !mbar_wait(&full[stage], phase, status)) *s_abort = 1;
        const uint32_t sA = base_u + stage * stage_bytes;
        const uint32_t sX = sA + 2 * kABytes;
        const int kb = ks * kKbPerStage + warp;  // this warp's k-block
        uint4 l0[2], l1[2], h0[2], h1[2];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            line_chunks(sA + t * kABytes, line_lo, tig, l0[t], l1[t]);
            line_chunks(sA + t * kABytes, line_hi, tig, h0[t], h1[t]);
        }
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            const int xr = n * 8 + g;  // activation row of this lane's B fragment
            uint4 x0 = make_uint4(0u, 0u, 0u, 0u), x1 = x0;
            xfrag(xr, kb, sX, x0, x1);
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                mma16816(acc[t][n], l0[t].x, h0[t].x, l0[t].y, h0[t].y, x0.x, x0.y);
                mma16816(acc[t][n], l0[t].z, h0[t].z, l0[t].w, h0[t].w, x0.z, x0.w);
                mma16816(acc[t][n], l1[t].x, h1[t].x, l1[t].y, h1[t].y, x1.x, x1.y);
                mma16816(acc[t][n], l1[t].z, h1[t].z, l1[t].w, h1[t].w, x1.z, x1.w);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
        if (++stage == depth) { stage = 0; phase ^= 1u; }
    }
}

// Sums the eight warps' accumulators of tile t in warp order and runs the
// epilogue for the R activation rows.  bar() synchronises the 256 consumer threads.
template <int NT, class Bar>
__device__ __forceinline__ void finish_tile(const MatvecArgs& e, const RowMap& rows, int t, int R,
                                            const float (&acc)[NT][4], float* red, Bar bar) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) red[((warp * NT + n) * 4 + i) * 32 + lane] = acc[n][i];
    bar();
    const mv::TileRows tr = tile_info(e, t);
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
        if (r0 < R) mv::epilogue(e, rows, tr, g, r0, v[0], v[2]);
        if (r0 + 1 < R) mv::epilogue(e, rows, tr, g, r0 + 1, v[1], v[3]);
    }
    bar();
}

// One whole tile t over its nst stages: accumulate_stages then finish_tile.
template <int NT, class XFrag, class Bar>
__device__ __forceinline__ void consume_tile(const MatvecArgs& e, const RowMap& rows, int t, int nst, int R,
                                             uint32_t base_u, int stage_bytes, int depth, int& stage, uint32_t& phase,
                                             uint64_t* full, uint64_t* empty, float* red, volatile int* s_abort,
                                             int* status, XFrag xfrag, Bar bar) {
    float acc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
    accumulate_stages<NT>(e, acc, 0, nst, base_u, stage_bytes, depth, stage, phase, full, empty, s_abort, status,
                          xfrag);
    finish_tile<NT>(e, rows, t, R, acc, red, bar);
}

// Activation rows (R rows of K bf16, row r at row(r), optionally RMSNormed
// with norm_w) into shared lines [k-block][row][64] (line l = kb * R + r, chunk
// c of line l at chunk c ^ (l mod 8)), by the 256 consumer threads.  The norm
// has the exact arithmetic of the standalone norm kernel.  red_norm: 8 floats
// per row.
template <class RowPtr, class Bar>
__device__ __forceinline__ void rows_to_lines(RowPtr row, const bf16* norm_w, float eps, int R, int K, uint32_t xs_u,
                                              float* red_norm, Bar bar) {
    const int tid = threadIdx.x;
    auto put = [&](int i, int r, const uint4& o) {
        const int line = (i >> 6) * R + r, c = (i & 63) >> 3;
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(xs_u + line * 128 + ((c ^ (line & 7)) << 4)),
                     "r"(o.x), "r"(o.y), "r"(o.z), "r"(o.w)
                     : "memory");
    };
    for (int r = 0; r < R; ++r) {
        const bf16* hr = row(r);
        const float rinv = norm_w ? rms_inv(hr, K, eps, tid, red_norm + r * 8, bar) : 0.f;
        for (int i = tid * 8; i < K; i += kNormThreads * 8) {
            uint4 o = *reinterpret_cast<const uint4*>(hr + i);
            if (norm_w) {
                const uint4 wv = __ldg(reinterpret_cast<const uint4*>(norm_w + i));
                const bf16* he = reinterpret_cast<const bf16*>(&o);
                const bf16* we = reinterpret_cast<const bf16*>(&wv);
                uint4 n;
                bf16* ne = reinterpret_cast<bf16*>(&n);
#pragma unroll
                for (int k = 0; k < 8; ++k) ne[k] = rms_apply(he[k], we[k], rinv);
                o = n;
            }
            put(i, r, o);
        }
    }
    bar();
}

}  // namespace mvc
}  // namespace tfl
