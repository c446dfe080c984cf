// The arithmetic of decode attention, shared by the split attention kernels and
// the persistent decode-step kernel so that both give the same bits.
//
// Block partial (one 128-key block at absolute positions, one KV head, a group
// of rows): eight warps; S = Q K^T with warp w owning keys 16w..16w+15, scale
// by log2(e)/sqrt(128) and causal mask, block row max over the warps, weights
// p = 2^(s - max) split into hi/lo bf16, row sums, then O = P V with warp w
// owning dims 16w..16w+15.  Written per (row, head): m_b, l_b and o_b.
// Merge: per (row, head), M = max_b m_b, then L = sum l_b 2^(m_b - M) and
// O = sum o_b 2^(m_b - M), each folded over eight block slices (slice i takes
// blocks i, i+8, ...) in block order and the slices added in slice order;
// out = bf16(O / L).
#pragma once

#include "common.cuh"
#include "warp_mma.cuh"

namespace tfl {
namespace attn {

constexpr int kWarps = 8;            // warps taking part (256 threads)
constexpr int kKB = kPage;           // keys per block
constexpr int kMaxPairs = 32;        // up to 4 rows x 8 heads: two m16 tiles
constexpr int kMergeSlices = 8;
constexpr float kScale = 0.12751743074640502f;  // log2(e) / sqrt(128)

// Rows of 128 bf16 (256 bytes, 16 chunks of 16 bytes) with chunk c of row r
// stored at chunk c ^ (r & 7): the eight rows an ldmatrix reads hit distinct
// banks without padding.  Returns an element index.
__device__ __forceinline__ int swz(int row, int col) {
    return row * kHeadDim + (((col >> 3) ^ (row & 7)) << 3) + (col & 7);
}

struct BlockGeom {
    int b, g;        // key block, KV head
    int r0, P, MT;   // first row of the group (call-wide index), pairs, m16 tiles of pairs
    int k0, nv;      // first key, keys of the block any row of the group sees
    int p_first;     // position of the group's first row
};

// One block partial.  q_u: shared address of the queries (kMaxPairs x 128 bf16,
// swz layout; pairs past P zero).  p_u: shared address for the weights (two
// kMaxPairs x 128 tiles, hi then lo, swz layout); it may alias the keys.
// kaddr(row, col) / vaddr(row, col): shared address of the 16-byte chunk of key
// (or value) row `row` holding dims col..col+7.  bar(): barrier of the eight
// warps.  values_ready(): makes the values visible (called after the weights
// are written, before P V).  wmax/wsum: kWarps x kMaxPairs floats each.
template <int G, class KA, class VA, class Bar, class VReady>
__device__ __forceinline__ void block_partial(const AttnDecodeArgs& a, const BlockGeom& bg, uint32_t q_u, uint32_t p_u,
                                              float (*wmax)[kMaxPairs], float (*wsum)[kMaxPairs], KA kaddr, VA vaddr,
                                              Bar bar, VReady values_ready) {
    using wm::ldsm_x4;
    using wm::ldsm_x4_t;
    using wm::mma16816;
    using wm::pack_bf16;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;  // threads 0..255
    const int gq = lane >> 2, tig = lane & 3;
    const int P = bg.P, MT = bg.MT, nv = bg.nv, k0 = bg.k0;

    // ---- S = Q K^T: warp w owns keys 16w .. 16w+15 (two n8 tiles) ----
    float sc[2][2][4];  // [m tile][n tile][fragment]
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) sc[mt][nt][0] = sc[mt][nt][1] = sc[mt][nt][2] = sc[mt][nt][3] = 0.f;
    {
        const int mrow = (lane & 7) + ((lane >> 3) & 1) * 8, mcol = (lane >> 4) * 8;  // A: matrices (r, k) quads
        const int krow = (lane & 7) + (lane >> 4) * 8, kcol = ((lane >> 3) & 1) * 8;  // B: keys x dims
#pragma unroll
        for (int ks = 0; ks < kHeadDim / 16; ++ks) {
            uint32_t bk[4];
            ldsm_x4(bk, kaddr(warp * 16 + krow, ks * 16 + kcol));
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                if (mt < MT) {
                    uint32_t aq[4];
                    ldsm_x4(aq, q_u + 2u * swz(mt * 16 + mrow, ks * 16 + mcol));
                    mma16816(sc[mt][0], aq, bk[0], bk[1]);
                    mma16816(sc[mt][1], aq, bk[2], bk[3]);
                }
            }
        }
    }
    // scale, mask, per-warp row maxima
    float mx[2][2];  // [m tile][row half]
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int p = mt * 16 + gq + h * 8;
            const int pos_row = bg.p_first + (p < P ? p / G : 0);
            float m = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int t = warp * 16 + nt * 8 + 2 * tig + e;
                    const bool vis = p < P && t < nv && k0 + t <= pos_row;
                    float& v = sc[mt][nt][h * 2 + e];
                    v = vis ? v * kScale : -INFINITY;
                    m = fmaxf(m, v);
                }
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
            mx[mt][h] = m;
        }
    }
    if (tig == 0) {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int h = 0; h < 2; ++h) wmax[warp][mt * 16 + gq + h * 8] = mx[mt][h];
    }
    bar();
    // block row maxima, weights, per-warp row sums, weights to shared memory
    float bmax[2][2];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int p = mt * 16 + gq + h * 8;
            float m = wmax[0][p];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) m = fmaxf(m, wmax[w][p]);
            bmax[mt][h] = m;
            float l = 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                float e0 = 0.f, e1 = 0.f;
                if (m != -INFINITY) {
                    e0 = exp2f(sc[mt][nt][h * 2 + 0] - m);
                    e1 = exp2f(sc[mt][nt][h * 2 + 1] - m);
                }
                l += e0;
                l += e1;
                const bf16 h0 = rn(e0), h1 = rn(e1);
                const bf16 l0 = rn(e0 - bf(h0)), l1 = rn(e1 - bf(h1));
                const int t = warp * 16 + nt * 8 + 2 * tig;
                const uint32_t hi = pack_bf16(h0, h1), lo = pack_bf16(l0, l1);
                asm volatile("st.shared.u32 [%0], %1;" ::"r"(p_u + 2u * swz(p, t)), "r"(hi) : "memory");
                asm volatile("st.shared.u32 [%0], %1;" ::"r"(p_u + 2u * (kMaxPairs * kHeadDim + swz(p, t))), "r"(lo)
                             : "memory");
            }
            l += __shfl_xor_sync(0xffffffffu, l, 1);
            l += __shfl_xor_sync(0xffffffffu, l, 2);
            if (tig == 0) wsum[warp][p] = l;
        }
    }
    values_ready();

    // ---- O = P V: warp w owns dims 16w .. 16w+15 (two n8 tiles) ----
    float oc[2][2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) oc[mt][nt][0] = oc[mt][nt][1] = oc[mt][nt][2] = oc[mt][nt][3] = 0.f;
    {
        const int mrow = (lane & 7) + ((lane >> 3) & 1) * 8, mcol = (lane >> 4) * 8;  // A: pairs x keys
        const int vrow = (lane & 7) + ((lane >> 3) & 1) * 8, vcol = (lane >> 4) * 8;  // B (trans): keys x dims
#pragma unroll 2
        for (int ks = 0; ks < kKB / 16; ++ks) {
            uint32_t bv[4];
            ldsm_x4_t(bv, vaddr(ks * 16 + vrow, warp * 16 + vcol));
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                if (mt < MT) {
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
                        uint32_t ap[4];
                        ldsm_x4(ap, p_u + 2u * (part * kMaxPairs * kHeadDim + swz(mt * 16 + mrow, ks * 16 + mcol)));
                        mma16816(oc[mt][0], ap, bv[0], bv[1]);
                        mma16816(oc[mt][1], ap, bv[2], bv[3]);
                    }
                }
            }
        }
    }

    // ---- partials: o (unnormalised), m, l per (row, head) ----
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int p = mt * 16 + gq + h * 8;
            if (mt < MT && p < P) {
                const int row = bg.r0 + p / G, head = bg.g * G + p % G;
                const size_t idx = ((size_t)row * a.n_q + head) * a.max_blocks + bg.b;
                float* po = a.po + idx * kHeadDim + warp * 16 + 2 * tig;
                *reinterpret_cast<float2*>(po) = make_float2(oc[mt][0][h * 2 + 0], oc[mt][0][h * 2 + 1]);
                *reinterpret_cast<float2*>(po + 8) = make_float2(oc[mt][1][h * 2 + 0], oc[mt][1][h * 2 + 1]);
                if (warp == 0 && tig == 0) {
                    float l = wsum[0][p];
#pragma unroll
                    for (int w = 1; w < kWarps; ++w) l += wsum[w][p];
                    a.pm[idx] = bmax[mt][h];
                    a.pl[idx] = l;
                }
            }
        }
    }
}

// Merge of (row, head) by T threads (T = 128 x a divisor of 8): thread tid owns
// dim tid % 128 and slices tid / 128 + j * (T / 128).  Shared scratch: wts
// (1,024 floats), red (T / 32 floats), so (8 x 128 floats), sl (8 floats).
// bar(): barrier of the T threads.
template <int T, class Bar>
__device__ __forceinline__ void merge(const AttnDecodeArgs& a, int row, int head, int tid, float* wts, float* red,
                                      float (*so)[kHeadDim], float* sl, Bar bar) {
    constexpr int kStep = T / kHeadDim;          // slice step
    constexpr int kPer = kMergeSlices / kStep;   // slices per thread
    const int d = tid & (kHeadDim - 1), s0 = tid / kHeadDim;
    const int s = row_stream(a.rows, row);
    const int pos = a.rows.pos0[s] + (row - a.rows.row_start[s]);
    const int nb = pos / kKB + 1;
    const size_t base = ((size_t)row * a.n_q + head) * a.max_blocks;

    float M = -INFINITY;
    for (int b = tid; b < nb; b += T) M = fmaxf(M, a.pm[base + b]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if ((tid & 31) == 0) red[tid >> 5] = M;
    bar();
    M = red[0];
#pragma unroll
    for (int w = 1; w < T / 32; ++w) M = fmaxf(M, red[w]);

    float O[kPer], L[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) O[j] = L[j] = 0.f;
    for (int c = 0; c < nb; c += 1024) {
        const int n = min(1024, nb - c);
        bar();
        for (int b = tid; b < n; b += T) wts[b] = exp2f(a.pm[base + c + b] - M);
        bar();
        const float* pl = a.pl + base + c;
        const float* po = a.po + (base + c) * kHeadDim + d;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            int b = s0 + j * kStep;
            for (; b + 7 * kMergeSlices < n; b += 8 * kMergeSlices) {
                float lv[8], ov[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    lv[u] = pl[b + u * kMergeSlices];
                    ov[u] = po[(size_t)(b + u * kMergeSlices) * kHeadDim];
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    L[j] = fmaf(lv[u], wts[b + u * kMergeSlices], L[j]);
                    O[j] = fmaf(ov[u], wts[b + u * kMergeSlices], O[j]);
                }
            }
            for (; b < n; b += kMergeSlices) {
                L[j] = fmaf(pl[b], wts[b], L[j]);
                O[j] = fmaf(po[(size_t)b * kHeadDim], wts[b], O[j]);
            }
        }
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        so[s0 + j * kStep][d] = O[j];
        if (d == 0) sl[s0 + j * kStep] = L[j];
    }
    bar();
    if (tid < kHeadDim) {
        float Ot = so[0][d], Lt = sl[0];
#pragma unroll
        for (int i = 1; i < kMergeSlices; ++i) {
            Ot += so[i][d];
            Lt += sl[i];
        }
        a.out[(size_t)row * a.n_q * kHeadDim + (size_t)head * kHeadDim + d] = rn(Ot / Lt);
    }
}

}  // namespace attn
}  // namespace tfl
