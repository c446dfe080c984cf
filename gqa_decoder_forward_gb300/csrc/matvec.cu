// Decode-row projections: y[r][n] = sum_k W[n][k] x[r][k] for 1..64 activation
// rows, fp32 sums rounded once to bf16, with the epilogue that follows the
// projection fused in (row projections of pull request #1415, section "How":
// "decode windows on ll_matvec with fp32 sums rounded once").
//
// HBM-bound: the weights are streamed exactly once per call with 16-byte
// loads that bypass L1 and carry an L2 evict-first hint; the activation rows
// (<= 64 x K bf16) stay L1/L2-resident.  The multiply runs on mma.sync
// m16n8k16 (bf16 in, fp32 accumulate): 16 weight rows form the A operand and
// up to 8 activation rows one n8 B tile.  A 16-byte load of 8 consecutive k of
// one weight row feeds two MMAs directly (no shared-memory staging): the k
// order inside each 32-wide chunk is permuted identically for A and B, which
// leaves every dot product unchanged.
//
// Determinism: the reduction order of an output depends only on (matrix, K):
// 8 warps own fixed K ranges, each accumulates its range in k order, and the
// 8 partials are added in warp order.  A row's result is therefore identical
// whether it is computed alone or beside 63 others (one-row steps == windows).
//
// A CTA owns a "tile" of 16 weight rows made of two groups of 8 (lo, hi),
// chosen so that the values an epilogue must combine meet in one thread:
//   STORE / RESIDUAL  rows 16t..16t+7 and 16t+8..16t+15
//   SWIGLU            gate rows 8t.. and up rows 8t..   (g and u of a feature)
//   QKV_ROPE          head h dims j0..j0+7 and j0+64..j0+71 (a NeoX RoPE pair)
#include "common.cuh"

namespace tfl {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint4 ld_weights(const bf16* p, uint64_t pol) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p), "l"(pol));
    return r;
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

struct TileRows {
    const bf16* lo;  // first of 8 consecutive weight rows (row g of the group = lo + g*K)
    const bf16* hi;
    int seg;         // QKV: 0 q, 1 k, 2 v
    int head;        // QKV: head within the segment
    int j0;          // QKV: first dim of the lo group (< 64); STORE/RESIDUAL: first row
};

__device__ __forceinline__ TileRows tile_rows(const MatvecArgs& a, int t) {
    TileRows r;
    const size_t K = (size_t)a.K;
    r.seg = 0;
    r.head = 0;
    r.j0 = 0;
    if (a.mode == MV_SWIGLU) {
        r.lo = a.w0 + (size_t)t * 8 * K;
        r.hi = a.w1 + (size_t)t * 8 * K;
        r.j0 = t * 8;
    } else if (a.mode == MV_QKV_ROPE) {
        int tq = a.n_q * 8, tk = a.n_kv * 8;
        const bf16* w;
        int u;
        if (t < tq) { r.seg = 0; w = a.w0; u = t; }
        else if (t < tq + tk) { r.seg = 1; w = a.w1; u = t - tq; }
        else { r.seg = 2; w = a.w2; u = t - tq - tk; }
        r.head = u / 8;
        r.j0 = (u % 8) * 8;
        r.lo = w + ((size_t)r.head * kHeadDim + r.j0) * K;
        r.hi = w + ((size_t)r.head * kHeadDim + 64 + r.j0) * K;
    } else {
        r.lo = a.w0 + (size_t)t * 16 * K;
        r.hi = r.lo + 8 * K;
        r.j0 = t * 16;
    }
    return r;
}

__device__ __forceinline__ float silu(float g) { return g / (1.0f + expf(-g)); }

// Epilogue of one (feature pair, activation row): vlo/vhi are the fp32 sums of
// the lo-group row g and the hi-group row g for activation row r.
__device__ __forceinline__ void epilogue(const MatvecArgs& a, const TileRows& tr, int g, int r, float vlo,
                                         float vhi) {
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
        const int s = row_stream(a.rows, r);
        const int pos = a.rows.pos0[s] + (r - a.rows.row_start[s]);
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
            bf16* row = kv_row(a.rows.kv[s], a.layer, tr.seg - 1, pos, a.n_kv) + (size_t)tr.head * kHeadDim;
            row[jl] = ol;
            row[jh] = oh;
        }
    }
}

template <int NT, int U>
__global__ void __launch_bounds__(kThreads, 2) matvec_kernel(const __grid_constant__ MatvecArgs a) {
    __shared__ float red[kWarps][NT][4][32];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tig = lane & 3;
    const TileRows tr = tile_rows(a, blockIdx.x);
    const int K = a.K;
    const int cpw = K / (32 * kWarps);  // 32-wide chunks per warp
    const int kb = warp * cpw * 32 + tig * 8;
    const bf16* plo = tr.lo + (size_t)g * K + kb;
    const bf16* phi = tr.hi + (size_t)g * K + kb;
    const uint64_t pol = evict_first_policy();

    // The first batch of weights does not depend on earlier kernels: issue it
    // before waiting for the producer of x.
    uint4 wl[U], wh[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        if (u < cpw) {
            wl[u] = ld_weights(plo + u * 32, pol);
            wh[u] = ld_weights(phi + u * 32, pol);
        }
    }
    pdl_wait();

    float acc[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;

    const bf16* xb = a.x + kb;
    for (int c = 0; c < cpw; c += U) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (c + u < cpw) {
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const int r = j * 8 + g;
                    uint4 xv = make_uint4(0u, 0u, 0u, 0u);
                    if (r < a.n_rows) xv = __ldg(reinterpret_cast<const uint4*>(xb + (size_t)r * K + (c + u) * 32));
                    mma16816(acc[j], wl[u].x, wh[u].x, wl[u].y, wh[u].y, xv.x, xv.y);
                    mma16816(acc[j], wl[u].z, wh[u].z, wl[u].w, wh[u].w, xv.z, xv.w);
                }
                if (c + U + u < cpw) {
                    wl[u] = ld_weights(plo + (c + U + u) * 32, pol);
                    wh[u] = ld_weights(phi + (c + U + u) * 32, pol);
                }
            }
        }
    }

#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) red[warp][j][i][lane] = acc[j][i];
    __syncthreads();
    pdl_trigger();

    // warp j finishes n8 tile j: partials added in warp order 0..7
    for (int j = warp; j < NT; j += kWarps) {
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float s = red[0][j][i][lane];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) s += red[w][j][i][lane];
            v[i] = s;
        }
        // c0 = (lo g, row 2tig), c1 = (lo g, row 2tig+1), c2 = (hi g, row 2tig), c3 = (hi g, row 2tig+1)
        const int r0 = j * 8 + 2 * tig;
        if (r0 < a.n_rows) epilogue(a, tr, g, r0, v[0], v[2]);
        if (r0 + 1 < a.n_rows) epilogue(a, tr, g, r0 + 1, v[1], v[3]);
    }
}

template <int NT, int U>
cudaError_t launch_nt(const MatvecArgs& a, int tiles, cudaStream_t st, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, matvec_kernel<NT, U>, a);
}

}  // namespace

int matvec_tiles(const MatvecArgs& a) {
    if (a.mode == MV_SWIGLU) return a.n_out / 8;
    if (a.mode == MV_QKV_ROPE) return (a.n_q + 2 * a.n_kv) * 8;
    return a.n_out / 16;
}

cudaError_t launch_matvec(const MatvecArgs& a, cudaStream_t st, bool pdl) {
    if (a.K % 256 != 0 || a.n_rows < 1 || a.n_rows > kMaxDecodeRows) return cudaErrorInvalidValue;
    const int tiles = matvec_tiles(a);
    if (a.n_rows <= 8) return launch_nt<1, 8>(a, tiles, st, pdl);
    if (a.n_rows <= 16) return launch_nt<2, 8>(a, tiles, st, pdl);
    if (a.n_rows <= 32) return launch_nt<4, 4>(a, tiles, st, pdl);
    return launch_nt<8, 4>(a, tiles, st, pdl);
}

}  // namespace tfl
