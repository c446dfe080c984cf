// Epilogues of the decode projections, shared by the matvec kernels: each
// lane finishes the fp32 sums of one feature pair (lo, hi) for one activation
// row and applies the op that follows the projection.
#pragma once

#include "common.cuh"

namespace tfl {
namespace mv {

struct TileRows {
    const bf16* lo;  // first of 8 consecutive weight rows (row g of the group = lo + g*K)
    const bf16* hi;
    int seg;         // QKV: 0 q, 1 k, 2 v
    int head;        // QKV: head within the segment
    int j0;          // QKV: first dim of the lo group (< 64); STORE/RESIDUAL: first row
};

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

// Epilogue of one (feature pair, activation row): vlo/vhi are the fp32 sums of
// the lo-group row g and the hi-group row g for activation row r.
__device__ __forceinline__ void epilogue(const MatvecArgs& a, const RowMap& rows, const TileRows& tr, int g, int r,
                                         float vlo, float vhi) {
    if (a.mode == MV_STORE) {
        bf16* y = a.y + (size_t)r * a.ldy + tr.j0;
        y[g] = rn(vlo);
        y[8 + g] = rn(vhi);
    } else if (a.mode == MV_RESIDUAL) {
        bf16* h = a.h + (size_t)r * a.n_out + tr.j0;
        h[g] = rn(bf(h[g]) + rbf(vlo));
        h[8 + g] = rn(bf(h[8 + g]) + rbf(vhi));
    } else if (a.mode == MV_SWIGLU) {
        float gate = rbf(vlo), up = rbf(vhi);
        a.y[(size_t)r * a.ldy + tr.j0 + g] = rn(rbf(silu(gate)) * up);
    } else {  // MV_QKV_ROPE
        const int jl = tr.j0 + g, jh = jl + 64;
        float xl = rbf(vlo), xh = rbf(vhi);
        const int s = row_stream(rows, r);
        const int pos = rows.pos0[s] + (r - rows.row_start[s]);
        bf16 ol, oh;
        if (tr.seg < 2) {
            float c = bf(a.cos_t[(size_t)pos * 64 + jl]);
            float sn = bf(a.sin_t[(size_t)pos * 64 + jl]);
            ol = rn(rbf(xl * c) + rbf(-xh * sn));
            oh = rn(rbf(xh * c) + rbf(xl * sn));
        } else {
            ol = rn(xl);
            oh = rn(xh);
        }
        if (tr.seg == 0) {
            bf16* q = a.y + (size_t)r * a.ldy + (size_t)tr.head * kHeadDim;
            q[jl] = ol;
            q[jh] = oh;
        } else {
            bf16* row = kv_row(rows.kv[s], a.layer, tr.seg - 1, pos, a.n_kv) + (size_t)tr.head * kHeadDim;
            row[jl] = ol;
            row[jh] = oh;
        }
    }
}


}  // namespace mv
}  // namespace tfl
