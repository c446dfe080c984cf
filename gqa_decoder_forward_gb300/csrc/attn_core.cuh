// The arithmetic of decode attention, shared by the split attention kernels and
// the persistent decode-step kernel so that both give the same bits.
//
// Unit partial (512 keys at absolute positions, one KV head, a group of up to
// two rows, or four in the kernel that serves streams of several rows): warp w of eight owns keys 16w..16w+15 of each 128-key sub-block
// and runs an online softmax over them (S = Q K^T scaled by log2(e)/sqrt(128)
// and causally masked, running max, weights p = 2^(s - max) split into hi/lo
// bf16, running sums, O = P V); the warp partials are then combined in warp
// order.  Written per (row, head): m_u, l_u and o_u.
// Merge: per (row, head), M = max_u m_u, then L = sum l_u 2^(m_u - M) and
// O = sum o_u 2^(m_u - M) folded in unit order over four contiguous quarters,
// the quarters added in order; out = bf16(O / L).
#pragma once

#include "common.cuh"
#include "warp_mma.cuh"

namespace tfl {
namespace attn {

constexpr int kWarps = 8;            // warps taking part (256 threads)
constexpr int kKB = kPage;           // keys per block
constexpr float kScale = 0.12751743074640502f;  // log2(e) / sqrt(128)
// A warp's reference max for a pair moves only when a sub-block's max exceeds
// it by more than kLazy (log2 units), so its weights stay <= 2^kLazy and the
// running output is rescaled only then.
constexpr float kLazy = 8.f;

// 2^x by the special-function unit (approximate, flushes subnormal results to
// zero; 2^-inf = 0).
__device__ __forceinline__ float exp2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Rows of 128 bf16 (256 bytes, 16 chunks of 16 bytes) with chunk c of row r
// stored at chunk c ^ (r & 7): the eight rows an ldmatrix reads hit distinct
// banks without padding.  Returns an element index.
__device__ __forceinline__ int swz(int row, int col) {
    return row * kHeadDim + (((col >> 3) ^ (row & 7)) << 3) + (col & 7);
}

// A unit is 512 keys at absolute positions (kUnit): up to four sub-blocks of
// 128 keys (one cache page each).  Warp w of the eight owns keys 16w..16w+15 of
// every sub-block and keeps its own running max, sum and output for the
// unit; the eight warp partials are combined once at the end, in warp order.
constexpr int kSub = kPage;          // keys per sub-block
constexpr int kUnit = kAttnUnit;     // keys per unit (one partial per (row, head, unit))
constexpr int kGroupRows = 2;        // rows per group: G * 2 <= 16 (row, head) pairs, two n8 tiles
constexpr int kPairs = 16;
// the cp.async kernel's groups: G * 4 <= 32 pairs, four n8 tiles (each pair's
// arithmetic is the same whatever the group; larger groups give each warp more
// independent accumulation chains and read each key block once per four rows)
constexpr int kWideGroupRows = 4;
constexpr int kWidePairs = 32;
// combine scratch per pair: the warps' outputs, maxima, sums and weights, and M.
// A warp's output row of a pair takes kCoStride floats (128 + 4: the two pairs a
// thread writes then fall in different banks)
constexpr int kCoStride = kHeadDim + 4;
constexpr int kCombPerPair = kWarps * kCoStride + 3 * kWarps + 1;
constexpr int kCombFloats = kCombPerPair * kPairs;  // 16 pairs
// floats of combine scratch for P pairs (the combine takes at most 16 pairs at a time)
__host__ __device__ constexpr int comb_floats(int P) { return kCombPerPair * ((((P < 16 ? P : 16) + 7) / 8) * 8); }

struct UnitGeom {
    int u, g;        // unit, KV head
    int r0, P;       // first row of the group (call-wide index), (row, head) pairs (<= 32)
    int k0;          // first key of the unit
    int nsub;        // sub-blocks holding keys any row of the group sees (1..4)
    int p_first, p_last;  // positions of the group's first and last rows
};

// The second half of the combine of one pass of up to PS pairs (pairs c0 * 8
// .. c0 * 8 + PP - 1 of the unit), once the eight warps' outputs, maxima and
// sums are in the scratch (co [warp][pair][dim] in rows of kCoStride, cm and
// cl [warp][pair], pair stride PS): one thread per (warp, pair) takes M = max_w m_w and
// a_w = 2^(m_w - M) into cw and cM, then thread (pair, dim) folds
// O = sum_w O_w a_w and L = sum_w l_w a_w in warp order and writes the unit's
// m_u = M, l_u = L and o_u = O.  Run by T threads (tid = 0..T-1, T a multiple
// of 32); bar() synchronises those T threads.
template <int G, int PS, int T, class Bar>
__device__ __forceinline__ void combine_pass(const AttnDecodeArgs& a, int r0, int g, int u, int c0, int PP,
                                             float* comb, int tid, Bar bar) {
    static_assert(T % 32 == 0, "combine threads");
    const float* co = comb;
    const float* cm = comb + kWarps * PS * kCoStride;
    const float* cl = cm + kWarps * PS;
    float* cw = const_cast<float*>(cl) + kWarps * PS;
    float* cM = cw + kWarps * PS;
    for (int i = tid; i < kWarps * PS; i += T) {
        const int w = i / PS, p = i % PS;
        if (p < PP) {
            float M = cm[p];
#pragma unroll
            for (int v = 1; v < kWarps; ++v) M = fmaxf(M, cm[v * PS + p]);
            const float mw = cm[w * PS + p];
            cw[w * PS + p] = (M == -INFINITY || mw == -INFINITY) ? 0.f : exp2f(mw - M);
            if (w == 0) cM[p] = M;
        }
    }
    bar();
    for (int i = tid; i < PP * kHeadDim; i += T) {  // (pair, dim) = (i / 128, i % 128)
        const int p = i / kHeadDim, d = i % kHeadDim;
        const float M = cM[p];
        float O = 0.f, L = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) O = fmaf(co[((size_t)w * PS + p) * kCoStride + d], cw[w * PS + p], O);
            if (d == 0) {
#pragma unroll
                for (int w = 0; w < kWarps; ++w) L = fmaf(cl[w * PS + p], cw[w * PS + p], L);
            }
        }
        const int pg = c0 * 8 + p;
        const int row = r0 + pg / G, head = g * G + pg % G;
        const size_t idx = ((size_t)row * a.n_q + head) * a.max_blocks + u;
        a.po[idx * kHeadDim + d] = O;
        if (d == 0) {
            a.pm[idx] = M;
            a.pl[idx] = L;
        }
    }
}

// One unit partial by the eight warps (threads 0..255).  q_u: shared address
// of the queries (8 NP pairs x 128 bf16, swz layout, pairs past P zero), visible
// to every warp.  comb: comb_floats(P) floats of shared memory.  src provides,
// for sub-block j: wait(j) (this warp may read the sub-block's keys and
// values; values past the last visible key are exact zeros), done(j) (this
// warp has read its last key and value of j), k(j, row, col) / v(j, row, col)
// (shared address of the 16-byte chunk of key / value row `row` holding dims
// col..col+7).  bar(): barrier of the eight warps.
//
// The products are taken transposed so that keys (and dims) fill the 16-row
// side of the m16n8k16 tensor-core shape and the (row, head) pairs the 8-wide
// side: S^T = K Q^T, then O^T += V^T P^T with P^T moved from the accumulator
// layout into the operand layout by an in-register transpose (movmatrix).
// Warp w, per pair and sub-block j, over its 16 keys: scores
// s = (q . k) log2(e)/sqrt(128) (masked: -inf), x = max s over the 16 keys;
// if x > m + kLazy the reference max moves: alpha = 2^(m - x), m = x, else
// alpha = 1; p = 2^(s - m) (<= 2^kLazy); per thread l_t = l_t alpha + (its two
// keys' p), O = O alpha (skipped when no pair of the warp moved: alpha = 1)
// + P V (hi part, then lo part); at the end of the unit l = the fixed shuffle
// tree of the eight l_t of the pair.  Combine: M = max_w m_w,
// a_w = 2^(m_w - M), L = sum_w l_w a_w, O = sum_w O_w a_w (fused multiply-adds
// in warp order).  A pair with no visible key keeps m = -inf, l = 0, O = 0.
// Up to two pair tiles the query fragments stay in registers for the unit;
// with more they are read from shared memory again at every sub-block (the
// same values, so the same products), and the combine runs in passes of two
// pair tiles.  pre() runs before the warps write into comb (it may wait until
// comb is free).  HANDOFF (at most two pair tiles): the warps only write their
// outputs, maxima and sums into comb and return; combine_pass, run by other
// threads once all eight warps have written, finishes the unit.
struct NoPre {
    __device__ __forceinline__ void operator()() const {}
};
template <int G, int NP, bool HANDOFF = false, class Src, class Bar, class Pre = NoPre>
__device__ __forceinline__ void unit_partial_np(const AttnDecodeArgs& a, const UnitGeom& ug, uint32_t q_u,
                                                float* comb, Src& src, Bar bar, Pre pre = Pre()) {
    static_assert(!HANDOFF || NP <= 2, "a hand-off holds one pass");
    using wm::ldsm_x4;
    using wm::ldsm_x4_t;
    using wm::mma16816;
    using wm::movmatrix_t;
    using wm::pack_bf16;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;  // threads 0..255
    const int gq = lane >> 2, tig = lane & 3;
    const int P = ug.P;  // NP = (P + 7) / 8 n8 tiles of pairs
    const int arow = (lane & 7) + ((lane >> 3) & 1) * 8, acol = (lane >> 4) * 8;  // A (non-trans): 16 x 16
    const int trow = (lane & 7) + (lane >> 4) * 8, tcol = ((lane >> 3) & 1) * 8;  // A (trans): 16 x 16

    // Q^T as B fragments: [n tile][k step][2]
    constexpr bool kQRegs = NP <= 2;
    constexpr int NQ = kQRegs ? NP : 1;
    uint32_t qb[NQ][kHeadDim / 16][2];
#pragma unroll
    for (int nt = 0; nt < NQ; ++nt) {
        if (kQRegs) {
#pragma unroll
            for (int ks = 0; ks < kHeadDim / 16; ks += 2) {
                uint32_t r[4];
                ldsm_x4(r, q_u + 2u * swz(nt * 8 + (lane & 7), ks * 16 + (lane >> 3) * 8));
                qb[nt][ks][0] = r[0];
                qb[nt][ks][1] = r[1];
                qb[nt][ks + 1][0] = r[2];
                qb[nt][ks + 1][1] = r[3];
            }
        }
    }
    // this thread's pairs: nt * 8 + 2 * tig + e
    int pos_p[NP][2];
#pragma unroll
    for (int nt = 0; nt < NP; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int p = nt * 8 + 2 * tig + e;
            pos_p[nt][e] = p < P ? ug.p_first + p / G : -1;  // -1: a padding pair sees nothing
        }
    float m_w[NP][2], l_w[NP][2];
    float ot[kHeadDim / 16][NP][4];  // [dim tile][pair tile][fragment]
#pragma unroll
    for (int nt = 0; nt < NP; ++nt) {
        m_w[nt][0] = m_w[nt][1] = -INFINITY;
        l_w[nt][0] = l_w[nt][1] = 0.f;
#pragma unroll
        for (int dt = 0; dt < kHeadDim / 16; ++dt) ot[dt][nt][0] = ot[dt][nt][1] = ot[dt][nt][2] = ot[dt][nt][3] = 0.f;
    }

    for (int j = 0; j < ug.nsub; ++j) {
        const int kj = ug.k0 + j * kSub;
        const int nv = min(kSub, ug.p_last + 1 - kj);  // keys of the sub-block any row sees
        src.wait(j);
        // ---- S^T = K Q^T: 16 keys (rows gq, gq+8) x 8 pairs per tile ----
        float st[NP][4];
#pragma unroll
        for (int nt = 0; nt < NP; ++nt) st[nt][0] = st[nt][1] = st[nt][2] = st[nt][3] = 0.f;
        if constexpr (kQRegs) {
#pragma unroll
            for (int ks = 0; ks < kHeadDim / 16; ++ks) {
                uint32_t ak[4];
                ldsm_x4(ak, src.k(j, warp * 16 + arow, ks * 16 + acol));
#pragma unroll
                for (int nt = 0; nt < NP; ++nt)
                    mma16816(st[nt], ak, qb[nt][ks][0], qb[nt][ks][1]);
            }
        } else {
#pragma unroll
            for (int ks = 0; ks < kHeadDim / 16; ks += 2) {
                uint32_t ak0[4], ak1[4];
                ldsm_x4(ak0, src.k(j, warp * 16 + arow, ks * 16 + acol));
                ldsm_x4(ak1, src.k(j, warp * 16 + arow, (ks + 1) * 16 + acol));
#pragma unroll
                for (int nt = 0; nt < NP; ++nt) {
                    uint32_t r[4];  // k steps ks and ks + 1 of pair tile nt
                    ldsm_x4(r, q_u + 2u * swz(nt * 8 + (lane & 7), ks * 16 + (lane >> 3) * 8));
                    mma16816(st[nt], ak0, r[0], r[1]);
                    mma16816(st[nt], ak1, r[2], r[3]);
                }
            }
        }
        // ---- per pair: reference max, weights, running sums; P^T operands ----
        // every row of the group sees every key of the sub-block: no masking
        const bool full_vis = kj + kSub - 1 <= ug.p_first;
        uint32_t pbh[NP][2], pbl[NP][2];  // [pair tile][keys 0-7 / 8-15]
#pragma unroll
        for (int nt = 0; nt < NP; ++nt) {
            float alpha[2], pe[2][2];  // pe[key half][pair e]
            bool moved = false;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float mx = -INFINITY;
#pragma unroll
                for (int hk = 0; hk < 2; ++hk) {
                    float& v = st[nt][hk * 2 + e];
                    if (full_vis) {
                        v *= kScale;
                    } else {
                        const int t = warp * 16 + gq + hk * 8;
                        const bool vis = t < nv && kj + t <= pos_p[nt][e];
                        v = vis ? v * kScale : -INFINITY;
                    }
                    mx = fmaxf(mx, v);
                }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                alpha[e] = 1.f;
                if (mx > m_w[nt][e] + kLazy) {  // also the first visible key (m = -inf)
                    alpha[e] = exp2_approx(m_w[nt][e] - mx);
                    m_w[nt][e] = mx;
                    moved = true;
                }
                const float m = m_w[nt][e];
#pragma unroll
                for (int hk = 0; hk < 2; ++hk)
                    pe[hk][e] = m == -INFINITY ? 0.f : exp2_approx(st[nt][hk * 2 + e] - m);
                l_w[nt][e] = fmaf(l_w[nt][e], alpha[e], pe[0][e] + pe[1][e]);
            }
#pragma unroll
            for (int hk = 0; hk < 2; ++hk) {
                const bf16 h0 = rn(pe[hk][0]), h1 = rn(pe[hk][1]);
                pbh[nt][hk] = movmatrix_t(pack_bf16(h0, h1));
                pbl[nt][hk] = movmatrix_t(pack_bf16(rn(pe[hk][0] - bf(h0)), rn(pe[hk][1] - bf(h1))));
            }
            if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
                for (int dt = 0; dt < kHeadDim / 16; ++dt) {
                    ot[dt][nt][0] *= alpha[0];
                    ot[dt][nt][1] *= alpha[1];
                    ot[dt][nt][2] *= alpha[0];
                    ot[dt][nt][3] *= alpha[1];
                }
            }
        }
        // ---- O^T += V^T P^T over this warp's 16 keys: 8 dim tiles ----
#pragma unroll
        for (int dt = 0; dt < kHeadDim / 16; ++dt) {
            uint32_t av[4];
            ldsm_x4_t(av, src.v(j, warp * 16 + trow, dt * 16 + tcol));
#pragma unroll
            for (int nt = 0; nt < NP; ++nt) {
                mma16816(ot[dt][nt], av, pbh[nt][0], pbh[nt][1]);
                mma16816(ot[dt][nt], av, pbl[nt][0], pbl[nt][1]);
            }
        }
        src.done(j);
    }

    // each pair's sum over the warp's keys: the eight threads' sums by a fixed tree
#pragma unroll
    for (int nt = 0; nt < NP; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float l = l_w[nt][e];
            l += __shfl_xor_sync(0xffffffffu, l, 4);
            l += __shfl_xor_sync(0xffffffffu, l, 8);
            l += __shfl_xor_sync(0xffffffffu, l, 16);
            l_w[nt][e] = l;
        }
    // ---- combine the eight warp partials (warp order), two pair tiles a pass ----
    constexpr int CT = NP < 2 ? NP : 2;                 // pair tiles per pass
    constexpr int PS = CT * 8;                          // pair stride of the scratch
    float* co = comb;                                   // [warp][pair][dim], rows of kCoStride
    float* cm = comb + kWarps * PS * kCoStride;         // [warp][pair]
    float* cl = cm + kWarps * PS;
    pre();
#pragma unroll
    for (int c0 = 0; c0 < NP; c0 += CT) {
        if (c0 > 0) bar();  // the previous pass is done with the scratch
#pragma unroll
        for (int nt = c0; nt < (c0 + CT < NP ? c0 + CT : NP); ++nt) {
            const int lt = nt - c0;
#pragma unroll
            for (int dt = 0; dt < kHeadDim / 16; ++dt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int p = lt * 8 + 2 * tig + e;
                    co[((size_t)warp * PS + p) * kCoStride + dt * 16 + gq] = ot[dt][nt][e];
                    co[((size_t)warp * PS + p) * kCoStride + dt * 16 + gq + 8] = ot[dt][nt][2 + e];
                }
            if (gq == 0) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    cm[warp * PS + lt * 8 + 2 * tig + e] = m_w[nt][e];
                    cl[warp * PS + lt * 8 + 2 * tig + e] = l_w[nt][e];
                }
            }
        }
        if (HANDOFF) return;
        bar();
        combine_pass<G, PS, kWarps * 32>(a, ug.r0, ug.g, ug.u, c0, min(PS, P - c0 * 8), comb, tid, bar);
    }
    bar();  // the combine scratch and the queries may be reused
}

// The unit partial for P pairs; MAXNP (2 or 4) bounds the pair tiles the
// caller's groups can need, so kernels of two-row groups compile no wider path.
template <int G, int MAXNP = 2, class Src, class Bar>
__device__ __forceinline__ void unit_partial(const AttnDecodeArgs& a, const UnitGeom& ug, uint32_t q_u, float* comb,
                                             Src& src, Bar bar) {
    static_assert(MAXNP == 2 || MAXNP == 4, "two or four pair tiles");
    if (ug.P <= 8)
        unit_partial_np<G, 1>(a, ug, q_u, comb, src, bar);
    else if (MAXNP == 2 || ug.P <= 16)
        unit_partial_np<G, 2>(a, ug, q_u, comb, src, bar);
    else if (ug.P <= 24)
        unit_partial_np<G, MAXNP == 2 ? 2 : 3>(a, ug, q_u, comb, src, bar);
    else
        unit_partial_np<G, MAXNP>(a, ug, q_u, comb, src, bar);
}

// Merge of (row, head) over its units: M = max_u m_u; the units are cut into
// four contiguous quarters [q nu/4, (q+1) nu/4); per quarter and dim,
// O_q = sum o_u 2^(m_u - M) and L_q = sum l_u 2^(m_u - M) as fused multiply-adds
// in unit order; O = ((O_0 + O_1) + O_2) + O_3, L likewise; out = bf16(O / L).
// The fold depends only on the row's position (its unit count).
constexpr int kQuarters = 4;

// Folds quarter q for dim d; returns (O_q, L_q).
__device__ __forceinline__ float2 merge_quarter(const AttnDecodeArgs& a, size_t base, int nu, float M, int q, int d) {
    const int u0 = q * nu / kQuarters, u1 = (q + 1) * nu / kQuarters;
    float O = 0.f, L = 0.f;
    int u = u0;
    for (; u + 8 <= u1; u += 8) {
        float mv[8], lv[8], ov[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            mv[i] = a.pm[base + u + i];
            lv[i] = a.pl[base + u + i];
            ov[i] = a.po[(base + u + i) * kHeadDim + d];
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float w = exp2f(mv[i] - M);
            L = fmaf(lv[i], w, L);
            O = fmaf(ov[i], w, O);
        }
    }
    for (; u < u1; ++u) {
        const float w = exp2f(a.pm[base + u] - M);
        L = fmaf(a.pl[base + u], w, L);
        O = fmaf(a.po[(base + u) * kHeadDim + d], w, O);
    }
    return make_float2(O, L);
}

// The merge of (row, head) by T threads (T = 256: quarters q and q+2 per thread;
// T = 512: one quarter per thread).  Shared scratch: red (T / 32 floats), part
// (kQuarters x 128 float2), and optionally stage (kMergeStageFloats, 16-byte
// aligned), which lets rows of up to 32 units fetch all their partials at
// once.  bar(): barrier of the T threads.
constexpr int kMergeStageFloats = 8 * kQuarters * (kHeadDim + 2);
template <int T, class Bar>
__device__ __forceinline__ void merge(const AttnDecodeArgs& a, int row, int head, int tid, float* red, float2* part,
                                      Bar bar, float* stage = nullptr) {
    static_assert(T == 256 || T == 512, "256 or 512 threads");
    const int d = tid & (kHeadDim - 1), q0 = tid / kHeadDim;
    const int s = row_stream(a.rows, row);
    const int pos = a.rows.pos0[s] + (row - a.rows.row_start[s]);
    const int nu = pos / kUnit + 1;
    const size_t base = ((size_t)row * a.n_q + head) * a.max_blocks;
    if (stage && nu <= 8 * kQuarters) {
        // up to 32 units: every partial of the (row, head) is copied into
        // shared memory at once (one round trip, no registers held), then
        // folded exactly as below
        float* so = stage;                   // [nu][128]
        float* sm = stage + nu * kHeadDim;   // [nu] m_u
        float* sl = sm + 8 * kQuarters;      // [nu] l_u
        for (int i = tid; i < nu * (kHeadDim / 4); i += T)
            wm::cp_async16_zfill(so + i * 4, a.po + base * kHeadDim + i * 4, true);
        wm::cp_async_commit();
        if (tid < nu)
            sm[tid] = a.pm[base + tid];
        else if (tid >= 32 && tid < 32 + nu)
            sl[tid - 32] = a.pl[base + tid - 32];
        wm::cp_async_wait_all();
        bar();
        float M = -INFINITY;
        for (int u = 0; u < nu; ++u) M = fmaxf(M, sm[u]);
        for (int q = q0; q < kQuarters; q += T / kHeadDim) {
            const int u1 = (q + 1) * nu / kQuarters;
            float O = 0.f, L = 0.f;
            for (int u = q * nu / kQuarters; u < u1; ++u) {
                const float w = exp2f(sm[u] - M);
                L = fmaf(sl[u], w, L);
                O = fmaf(so[u * kHeadDim + d], w, O);
            }
            part[q * kHeadDim + d] = make_float2(O, L);
        }
    } else {
        float M = -INFINITY;
        for (int u = tid; u < nu; u += T) M = fmaxf(M, a.pm[base + u]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        if ((tid & 31) == 0) red[tid >> 5] = M;
        bar();
        M = red[0];
#pragma unroll
        for (int w = 1; w < T / 32; ++w) M = fmaxf(M, red[w]);
        for (int q = q0; q < kQuarters; q += T / kHeadDim)
            part[q * kHeadDim + d] = merge_quarter(a, base, nu, M, q, d);
    }
    bar();
    if (tid < kHeadDim) {
        float O = part[d].x, L = part[d].y;
#pragma unroll
        for (int q = 1; q < kQuarters; ++q) {
            O += part[q * kHeadDim + d].x;
            L += part[q * kHeadDim + d].y;
        }
        a.out[(size_t)row * a.n_q * kHeadDim + (size_t)head * kHeadDim + d] = rn(O / L);
    }
    bar();  // the scratch may be reused
}

}  // namespace attn
}  // namespace tfl
