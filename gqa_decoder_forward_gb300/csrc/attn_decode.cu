// Decode attention: causal GQA of a few rows per stream over a position-major
// paged bf16 cache, split over key units at absolute positions (pull request
// #1415, section "How": "decode rows on sdpa_vector lanes over key blocks at
// absolute positions").
//
// Pass 1 (attn_block_kernel): one CTA per (unit u of 512 positions, KV head g,
// group of <= 4 rows of one stream).  The unit's four 128-key sub-blocks of
// head g stream through two shared-memory buffers (cp.async), one computed
// while the next lands.  The G = n_q/n_kv query heads of the group's rows form
// the M dimension of tensor-core products (mma.sync m16n8k16, bf16 in, fp32
// accumulate); warp w owns keys 16w..16w+15 of every sub-block and runs its
// own online softmax (S = Q K^T, running max, O += P V), the warp partials are
// combined at the end.  Per (row, head) the CTA writes the unit's max score
// m_u, sum l_u = sum exp(s - m_u) and o_u = sum exp(s - m_u) v (attn_core.cuh).
// attn_block_tma_kernel computes the same partials with at most one persistent
// CTA per SM walking the (unit, KV head, row group) items in a fixed stride: a
// producer warp streams each item's sub-blocks as 16 KB TMA boxes (keys or
// values, 64 dims, 128-byte swizzle) through a 9-stage ring, each compute warp
// releases a stage once it has read its keys there, the next item's queries
// are copied during the last sub-block, and the eight warp partials of each
// unit go to a separate combine warpgroup through two shared buffers.
// Pass 2 (attn_merge_kernel): per (row, head), M = max_u m_u, then
// L = sum_u l_u e^(m_u - M) and O = sum_u o_u e^(m_u - M) in unit order,
// out = bf16(O / L).
//
// Precision: scores are fp32 dot products of the bf16 q and k, scaled in fp32;
// softmax weights are fp32 and enter P V as a pair of bf16 numbers
// (hi = bf16(p), lo = bf16(p - hi)), i.e. with about 16 significant bits --
// the weights are not rounded to bf16.
//
// Determinism: every row's arithmetic depends only on its own position: the
// unit and sub-block split is fixed by absolute position, masked keys have
// weight exactly 0 (a sub-block past a row leaves its running values
// unchanged), keys past the last one any row of the group sees are zero-filled
// in shared memory, and each output element of an mma depends only on its own
// row of P.  A row gives the same bits alone or beside other rows (one-row
// steps == windows, solo == batched).
#include <algorithm>

#include "common.cuh"
#include "attn_core.cuh"
#include "attn_decode.cuh"
#include "tma.cuh"
#include "warp_mma.cuh"

namespace tfl {
namespace {

constexpr int kThreads = 256;
constexpr int kRB = attn::kWideGroupRows;  // rows per CTA of attn_block_kernel
constexpr int kSub = attn::kSub;
constexpr int kUnit = attn::kUnit;
using attn::swz;

// 206,400 bytes (one CTA per SM): queries, two buffers of one sub-block's
// keys and values each (sub-block j+1 streams in while j is computed), and the
// scratch that combines the eight warp partials (16 pairs at a time).
struct Smem {
    bf16 q[attn::kWidePairs * kHeadDim];  // 8 KB
    bf16 k[2][kSub * kHeadDim];          // 2 x 32 KB
    bf16 v[2][kSub * kHeadDim];          // 2 x 32 KB
    float comb[attn::kCombFloats];       // 65 KB
};

using wm::cp_async16_zfill;
using wm::cp_async_commit;
using wm::cp_async_wait;

// Locates row group z of groups of rb rows: stream s, first row (global
// index) r0, row count nr.
__device__ __forceinline__ bool find_group(const RowMap& m, int z, int rb, int& s, int& r0, int& nr) {
    for (int t = 0; t < m.n_streams; ++t) {
        int rows = m.row_start[t + 1] - m.row_start[t];
        int ng = (rows + rb - 1) / rb;
        if (z < ng) {
            s = t;
            r0 = m.row_start[t] + z * rb;
            nr = min(rb, rows - z * rb);
            return true;
        }
        z -= ng;
    }
    return false;
}

// Sub-block staging through cp.async, two buffers (see attn::unit_partial for
// the contract): sub-block j lands in buffer j % 2 as one copy group; keys
// past the last visible one are zero-filled.
struct CpSrc {
    Smem* sm;
    const KvView* kv;
    int layer, n_kv, g, k0, p_last, nsub, issued;
    __device__ __forceinline__ void load(int j) {
        const int kj = k0 + j * kSub;
        const int nv = min(kSub, p_last + 1 - kj);
        const bf16* kbase = kv_row(*kv, layer, 0, kj, n_kv) + (size_t)g * kHeadDim;
        const bf16* vbase = kv_row(*kv, layer, 1, kj, n_kv) + (size_t)g * kHeadDim;
        const size_t pstride = (size_t)n_kv * kHeadDim;
        bf16* kd = sm->k[j & 1];
        bf16* vd = sm->v[j & 1];
        for (int i = threadIdx.x; i < kSub * 16; i += kThreads) {
            const int t = i >> 4, c = i & 15;
            const bool valid = t < nv;
            const size_t off = valid ? t * pstride + c * 8 : 0;
            cp_async16_zfill(kd + swz(t, c * 8), kbase + off, valid);
            cp_async16_zfill(vd + swz(t, c * 8), vbase + off, valid);
        }
        cp_async_commit();
        ++issued;
    }
    __device__ __forceinline__ uint32_t k(int j, int row, int col) const {
        return smem_u32(sm->k[j & 1]) + 2u * swz(row, col);
    }
    __device__ __forceinline__ uint32_t v(int j, int row, int col) const {
        return smem_u32(sm->v[j & 1]) + 2u * swz(row, col);
    }
    __device__ __forceinline__ void wait(int j) {
        if (issued > j + 1)
            cp_async_wait<1>();
        else
            cp_async_wait<0>();
        __syncthreads();
    }
    __device__ __forceinline__ void done(int j) {
        if (j + 2 < nsub) {
            __syncthreads();  // every warp is done with buffer j % 2
            load(j + 2);
        }
    }
};

// G = query heads per KV head.  Pair p = i*G + j is (row i of the group, head g*G + j).
template <int G>
__global__ void __launch_bounds__(kThreads, 1) attn_block_kernel(const __grid_constant__ AttnDecodeArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem& sm = *reinterpret_cast<Smem*>(smem_raw);

    int s, r0, nr;
    if (!find_group(a.rows, blockIdx.z, kRB, s, r0, nr)) return;
    const int u = blockIdx.x, g = blockIdx.y;
    const int p_first = a.rows.pos0[s] + (r0 - a.rows.row_start[s]);
    const int p_last = p_first + nr - 1;
    const int k0 = u * kUnit;
    if (k0 > p_last) return;
    const int tid = threadIdx.x;
    const int P = nr * G;  // (row, head) pairs, at most 32

    CpSrc src;
    src.sm = &sm;
    src.kv = &a.rows.kv[s];
    src.layer = a.layer;
    src.n_kv = a.n_kv;
    src.g = g;
    src.k0 = k0;
    src.p_last = p_last;
    src.nsub = min(4, (p_last - k0) / kSub + 1);
    src.issued = 0;
    // A unit whose keys all precede the stream's first row of this call holds
    // cache rows written by earlier calls (every kernel of the library signals
    // its dependents only after its own dependency wait, so those writers have
    // completed): its first sub-blocks stream in while the previous kernel is
    // still finishing.
    const bool early = k0 + src.nsub * kSub <= a.rows.pos0[s];
    if (early) {
        src.load(0);
        if (src.nsub > 1) src.load(1);
    }
    pdl_wait();
    pdl_trigger();
    if (!early) {
        src.load(0);
        if (src.nsub > 1) src.load(1);
    }
    // queries (bf16, unscaled); pairs past P are zero
    for (int i = tid; i < attn::kWidePairs * 16; i += kThreads) {
        const int p = i >> 4, c = i & 15;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (p < P) {
            const int row = r0 + p / G, head = g * G + p % G;
            val = *reinterpret_cast<const uint4*>(a.q + (size_t)row * a.n_q * kHeadDim + (size_t)head * kHeadDim +
                                                   c * 8);
        }
        *reinterpret_cast<uint4*>(&sm.q[swz(p, c * 8)]) = val;
    }
    __syncthreads();  // the queries
    attn::UnitGeom ug;
    ug.u = u;
    ug.g = g;
    ug.r0 = r0;
    ug.P = P;
    ug.k0 = k0;
    ug.nsub = src.nsub;
    ug.p_first = p_first;
    ug.p_last = p_last;
    attn::unit_partial<G, 4>(a, ug, smem_u32(sm.q), sm.comb, src, [] { __syncthreads(); });
}

// ---- TMA-fed variant -------------------------------------------------------------

// Four warpgroups: warps 0-7 compute the unit partials, warps 8-11 combine
// them, warp 12 is the TMA producer (13-15 idle).  The compute warps hand each
// unit's eight warp partials to the combine warps through a shared buffer and
// go on to the next unit (they wait for the buffer only when they are about to
// write the next unit's partials, a unit later), so the combine and its
// barriers no longer stall the stream.  setmaxnreg moves registers from the
// producer and combine warpgroups to the compute warps.
constexpr int kTConsumerWarps = 8;
constexpr int kTCombineWarps = 4;
constexpr int kTThreads = 16 * 32;
constexpr int kTRegsCompute = 168, kTRegsCombine = 112, kTRegsProducer = 56;
static_assert(128 * (2 * kTRegsCompute + kTRegsCombine + kTRegsProducer) <= kTThreads * 128,
              "register split exceeds the launch's registers");
// One-row streams only: an item has at most 8 (row, head) pairs, so a combine
// buffer is that of 8 pairs.
constexpr int kTDepth = 11;                            // ring stages
constexpr int kTCombFloats = attn::comb_floats(8);
constexpr int kTStage = kSub * 64 * 2;                 // 16 KB: 128 positions x 64 dims
constexpr int kTOffQ = kTDepth * kTStage;              // two query buffers (4 KB each)
constexpr int kTOffComb = kTOffQ + 2 * attn::kPairs * kHeadDim * 2;  // the combine buffer
constexpr int kTOffGeom = kTOffComb + kTCombFloats * 4;             // its unit's (r0, g, u, P)
constexpr int kTOffBar = kTOffGeom + 16;
constexpr int kTSmem = 1024 + kTOffBar + (2 * kTDepth + 2) * 8 + 16;
static_assert(kSub == kPage, "a sub-block is one cache page");
static_assert(kTSmem <= 227 * 1024, "shared memory");
static_assert((kTCombFloats * 4) % 16 == 0, "combine buffer alignment");

// A work item: unit u of KV head g for the group of rows r0 .. r0+nr-1 of stream s.
struct Item {
    int s, r0, nr, u, g, k0, nsub, p_first, p_last;
};

// Item w of the (group, KV head, unit) space, unit fastest; false when the unit
// holds no key any row of the group sees.
__device__ __forceinline__ bool item_at(const AttnDecodeArgs& a, int w, int nblk, Item& it) {
    it.u = w % nblk;
    const int rest = w / nblk;
    it.g = rest % a.n_kv;
    if (!find_group(a.rows, rest / a.n_kv, attn::kGroupRows, it.s, it.r0, it.nr)) return false;
    it.p_first = a.rows.pos0[it.s] + (it.r0 - a.rows.row_start[it.s]);
    it.p_last = it.p_first + it.nr - 1;
    it.k0 = it.u * kUnit;
    if (it.k0 > it.p_last) return false;
    it.nsub = min(4, (it.p_last - it.k0) / kSub + 1);
    return true;
}

// The first item at or after w (in steps of the grid) holding keys; W if none.
__device__ __forceinline__ int next_item(const AttnDecodeArgs& a, int w, int W, int nblk, Item& it) {
    for (; w < W; w += gridDim.x)
        if (item_at(a, w, nblk, it)) return w;
    return W;
}

struct TRing {
    int stage;
    uint32_t phase;
    __device__ __forceinline__ void advance() {
        if (++stage == kTDepth) {
            stage = 0;
            phase ^= 1u;
        }
    }
};

// Query (row, head) pair p of item it, 16-byte chunk c.
template <int G>
__device__ __forceinline__ const bf16* q_chunk(const AttnDecodeArgs& a, const Item& it, int p, int c) {
    const int row = it.r0 + p / G, head = it.g * G + p % G;
    return a.q + (size_t)row * a.n_q * kHeadDim + (size_t)head * kHeadDim + c * 8;
}

// Sub-block source over the ring (see attn::unit_partial): sub-block j of the
// item is the four stages after the item's first (K dims 0-63, K 64-127, V
// 0-63, V 64-127).  After the last sub-block, the next item's queries are
// copied (cp.async, one 16-byte chunk per consumer thread) into the other
// query buffer.
template <int G>
struct TmaSrc {
    unsigned char* base;
    uint64_t *full, *empty;
    TRing first;  // the item's first stage
    int* status;
    volatile int* abort;
    int k0, p_last, nsub;
    int stage[4];
    uint32_t sa[4];
    const AttnDecodeArgs* a;
    const Item* nx;  // null: no next item
    bf16* nq;        // the next item's query buffer
    __device__ __forceinline__ TRing at(int i) const {
        TRing r;
        const int t = first.stage + i;
        r.stage = t % kTDepth;
        r.phase = first.phase ^ (uint32_t)((t / kTDepth) & 1);
        return r;
    }
    __device__ __forceinline__ static uint32_t tile(uint32_t lo, uint32_t hi, int row, int col) {
        return (col < 64 ? lo : hi) + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4);
    }
    __device__ __forceinline__ uint32_t k(int, int row, int col) const { return tile(sa[0], sa[1], row, col); }
    __device__ __forceinline__ uint32_t v(int, int row, int col) const { return tile(sa[2], sa[3], row, col); }
    // this warp's key rows 16w..16w+15: values past the last visible key become
    // exact zeros (their weight is 0, and the cache there holds anything)
    __device__ __forceinline__ void wait(int j) {
        for (int i = 0; i < 4; ++i) {
            const TRing r = at(4 * j + i);
            stage[i] = r.stage;
            sa[i] = smem_u32(base + r.stage * kTStage);
            if (!*abort && !mbar_wait(&full[r.stage], r.phase, status)) *abort = 1;
        }
        const int nv = min(kSub, p_last + 1 - (k0 + j * kSub));
        const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const int r0 = max(nv, w * 16), r1 = w * 16 + 16;
        if (r0 < r1) {
            for (int i = lane; i < (r1 - r0) * 8 * 2; i += 32) {
                const int half = i >= (r1 - r0) * 8;
                const int c = half ? i - (r1 - r0) * 8 : i;
                asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"((half ? sa[3] : sa[2]) + r0 * 128 + c * 16),
                             "r"(0u)
                             : "memory");
            }
            // the stage is refilled by TMA later: order these generic writes before it
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
        }
    }
    __device__ __forceinline__ void done(int j) {
        __syncwarp();
        if ((threadIdx.x & 31) == 0)
            for (int i = 0; i < 4; ++i) mbar_arrive(&empty[stage[i]]);
        if (j == nsub - 1 && nx) {
            const int p = threadIdx.x >> 4, c = threadIdx.x & 15, P = nx->nr * G;
            cp_async16_zfill(&nq[swz(p, c * 8)], p < P ? q_chunk<G>(*a, *nx, p, c) : a->q, p < P);
            cp_async_commit();
        }
    }
};

struct TConsumerBar {
    __device__ __forceinline__ void operator()() const { named_barrier(1, kTConsumerWarps * 32); }
};

template <int G>
__global__ void __launch_bounds__(kTThreads, 1) attn_block_tma_kernel(const __grid_constant__ AttnDecodeArgs a,
                                                                      const __grid_constant__ KvMaps maps, int nblk,
                                                                      int W, int* status) {
    static_assert(attn::kPairs * 16 == kTConsumerWarps * 32, "one query chunk per consumer thread");
    extern __shared__ unsigned char smem_raw[];
    unsigned char* base =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(base + kTOffBar);
    uint64_t* empty = full + kTDepth;
    uint64_t* cfull = empty + kTDepth;  // the combine buffer holds the eight warps' partials
    uint64_t* cempty = cfull + 1;       // the combine warps are done with it
    volatile int* abort = reinterpret_cast<volatile int*>(cempty + 1);
    bf16* qbuf = reinterpret_cast<bf16*>(base + kTOffQ);
    float* comb = reinterpret_cast<float*>(base + kTOffComb);
    int4* geom = reinterpret_cast<int4*>(base + kTOffGeom);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    Item it;
    const int w0 = next_item(a, blockIdx.x, W, nblk, it);
    if (w0 >= W) return;  // uniform: no item for this CTA
    if (tid == 0) {
        for (int i = 0; i < kTDepth; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kTConsumerWarps);
        }
        mbar_init(cfull, kTConsumerWarps);
        mbar_init(cempty, 1);
        *abort = 0;
        mbar_init_fence();
    }
    __syncthreads();

    if (warp >= kTConsumerWarps + kTCombineWarps) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kTRegsProducer));
        // ---- producer: every item's sub-blocks in the consumers' order ----
        if (warp == kTConsumerWarps + kTCombineWarps && lane == 0) {
            const uint64_t pol = policy_evict_first();
            TRing rp{0, 0u};
            long long issued = 0;
            bool waited = false;
            for (int w = w0; w < W && !*abort; w = next_item(a, w + gridDim.x, W, nblk, it)) {
                // an item whose keys all precede the stream's first row of this
                // call holds cache rows written by earlier calls (every kernel of
                // the library signals its dependents only after its own
                // dependency wait): it streams in while the previous kernel ends
                if (!waited && it.k0 + it.nsub * kSub > a.rows.pos0[it.s]) {
                    pdl_wait();
                    waited = true;
                }
                const KvView& kv = a.rows.kv[it.s];
                for (int j = 0; j < it.nsub && !*abort; ++j) {
                    const int page = __ldg(kv.table + it.k0 / kPage + j);
                    for (int part = 0; part < 4; ++part) {  // K dims 0-63, K 64-127, V 0-63, V 64-127
                        if (!mbar_wait(&empty[rp.stage], rp.phase ^ 1u, status)) {
                            *abort = 1;
                            break;
                        }
                        mbar_arrive_expect_tx(&full[rp.stage], kTStage);
                        const int row0 = ((a.layer * 2 + (part >> 1)) * kv.n_pages + page) * kPage;
                        tma_load_3d(base + rp.stage * kTStage, &maps.m[it.s], (part & 1) * 64, it.g, row0,
                                    &full[rp.stage], pol);
                        ++issued;
                        rp.advance();
                    }
                }
            }
            // after an abort, the copies already issued land before the CTA exits
            if (*abort) drain_ring(full, kTDepth, rp.stage, rp.phase, issued, status);
        } else {
            pdl_wait();
            pdl_trigger();
        }
        return;
    }
    if (warp >= kTConsumerWarps) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kTRegsCombine));
        // ---- combine warps: each unit's warp partials, in the compute order ----
        pdl_wait();
        pdl_trigger();
        const int ct = tid - kTConsumerWarps * 32;
        auto cbar = [] { named_barrier(2, kTCombineWarps * 32); };
        uint32_t use = 0u;
        for (int w = w0; w < W; w = next_item(a, w + gridDim.x, W, nblk, it)) {
            const bool ok = mbar_wait_or_abort(cfull, use & 1u, abort, status);
            if (!named_barrier_and(2, kTCombineWarps * 32, ok)) break;  // every combine thread stops together
            const int4 gm = *geom;
            attn::combine_pass<G, 8, kTCombineWarps * 32>(a, gm.x, gm.y, gm.z, 0, gm.w, comb, ct, cbar);
            cbar();  // every combine thread is done with the buffer
            if (ct == 0) mbar_arrive(cempty);
            ++use;
        }
        return;
    }
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kTRegsCompute));
    // ---- compute warps: the eight warps of attn::unit_partial ----
    pdl_wait();
    pdl_trigger();
    for (int i = tid; i < attn::kPairs * 16; i += kTConsumerWarps * 32) {  // the first item's queries
        const int p = i >> 4, c = i & 15;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (p < it.nr * G) val = *reinterpret_cast<const uint4*>(q_chunk<G>(a, it, p, c));
        *reinterpret_cast<uint4*>(&qbuf[swz(p, c * 8)]) = val;
    }
    TConsumerBar bar;
    bar();
    TRing first{0, 0u};
    int w = w0, qb = 0;
    uint32_t use = 0u;
    for (;;) {
        Item nx;
        const int wn = next_item(a, w + gridDim.x, W, nblk, nx);
        TmaSrc<G> src;
        src.base = base;
        src.full = full;
        src.empty = empty;
        src.first = first;
        src.status = status;
        src.abort = abort;
        src.k0 = it.k0;
        src.p_last = it.p_last;
        src.nsub = it.nsub;
        src.a = &a;
        src.nx = wn < W ? &nx : nullptr;
        src.nq = qbuf + (qb ^ 1) * attn::kPairs * kHeadDim;
        attn::UnitGeom ug;
        ug.u = it.u;
        ug.g = it.g;
        ug.r0 = it.r0;
        ug.P = it.nr * G;
        ug.k0 = it.k0;
        ug.nsub = it.nsub;
        ug.p_first = it.p_first;
        ug.p_last = it.p_last;
        // one-row items: at most 8 (row, head) pairs, one pair tile; the
        // partials are written once the combine warps are done with the
        // previous unit's
        attn::unit_partial_np<G, 1, true>(a, ug, smem_u32(qbuf + qb * attn::kPairs * kHeadDim), comb, src, bar,
                                          [&] {
                                              if (!*abort && !mbar_wait_or_abort(cempty, (use & 1u) ^ 1u, abort, status))
                                                  *abort = 1;
                                          });
        if (tid == 0) *geom = make_int4(ug.r0, ug.g, ug.u, ug.P);
        __syncwarp();
        if (lane == 0) mbar_arrive(cfull);
        ++use;
        if (wn >= W) break;
        for (int i = 0; i < 4 * it.nsub; ++i) first.advance();
        it = nx;
        w = wn;
        qb ^= 1;
        cp_async_wait<0>();
        // the next item's queries; after an abort every compute thread stops here together
        if (named_barrier_or(1, kTConsumerWarps * 32, *abort != 0)) break;
    }
}

// One CTA of 512 threads (a quarter of the units per 128) per (head, row).
__global__ void __launch_bounds__(512) attn_merge_kernel(const __grid_constant__ AttnDecodeArgs a) {
    __shared__ float red[512 / 32];
    __shared__ float2 part[attn::kQuarters * kHeadDim];
    pdl_wait();
    pdl_trigger();
    attn::merge<512>(a, blockIdx.y, blockIdx.x, threadIdx.x, red, part, [] { __syncthreads(); });
}

}  // namespace

cudaError_t init_attn_decode() {
    cudaError_t e = cudaFuncSetAttribute(attn_block_kernel<7>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sizeof(Smem));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(attn_block_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(Smem));
}

cudaError_t init_attn_decode_tma() {
    cudaError_t e = cudaFuncSetAttribute(attn_block_tma_kernel<7>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTSmem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(attn_block_tma_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTSmem);
}

// Key blocks of the call; *groups = row groups of rb rows.
int attn_decode_blocks(const AttnDecodeArgs& a, int rb, int* groups) {
    int g = 0, max_pos = 0;
    for (int s = 0; s < a.rows.n_streams; ++s) {
        int rows = a.rows.row_start[s + 1] - a.rows.row_start[s];
        g += (rows + rb - 1) / rb;
        max_pos = max(max_pos, a.rows.pos0[s] + rows - 1);
    }
    *groups = g;
    return max_pos / kUnit + 1;
}

cudaError_t launch_attn_block(const AttnDecodeArgs& a, cudaStream_t st, bool pdl) {
    const int G = a.n_q / a.n_kv;
    if ((G != 7 && G != 8) || a.n_q % a.n_kv != 0) return cudaErrorInvalidValue;
    int groups = 0;
    const int nblk = attn_decode_blocks(a, kRB, &groups);
    if (nblk > a.max_blocks) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t c1 = {};
    c1.gridDim = dim3(nblk, a.n_kv, groups);
    c1.blockDim = dim3(kThreads);
    c1.dynamicSmemBytes = (int)sizeof(Smem);
    c1.stream = st;
    c1.attrs = attr;
    c1.numAttrs = pdl ? 1 : 0;
    return G == 7 ? cudaLaunchKernelEx(&c1, attn_block_kernel<7>, a) : cudaLaunchKernelEx(&c1, attn_block_kernel<8>, a);
}

cudaError_t launch_attn_block_tma(const AttnDecodeArgs& a, const KvMaps& maps, int* status, int sms,
                                  cudaStream_t st, bool pdl) {
    const int G = a.n_q / a.n_kv;
    if ((G != 7 && G != 8) || a.n_q % a.n_kv != 0 || sms < 1) return cudaErrorInvalidValue;
    for (int s = 0; s < a.rows.n_streams; ++s)  // the combine scratch holds one row's pairs
        if (a.rows.row_start[s + 1] - a.rows.row_start[s] != 1) return cudaErrorInvalidValue;
    int groups = 0;
    const int nblk = attn_decode_blocks(a, attn::kGroupRows, &groups);
    if (nblk > a.max_blocks) return cudaErrorInvalidValue;
    // one CTA per SM of the model's device at most (the shared memory holds one)
    const int W = nblk * a.n_kv * groups;  // work items
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t c = {};
    c.gridDim = dim3(std::min(W, sms));
    c.blockDim = dim3(kTThreads);
    c.dynamicSmemBytes = kTSmem;
    c.stream = st;
    c.attrs = attr;
    c.numAttrs = pdl ? 1 : 0;
    return G == 7 ? cudaLaunchKernelEx(&c, attn_block_tma_kernel<7>, a, maps, nblk, W, status)
                  : cudaLaunchKernelEx(&c, attn_block_tma_kernel<8>, a, maps, nblk, W, status);
}

cudaError_t launch_attn_merge(const AttnDecodeArgs& a, cudaStream_t st, bool pdl) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t c2 = {};
    c2.gridDim = dim3(a.n_q, a.rows.n_rows);
    c2.blockDim = dim3(512);
    c2.stream = st;
    c2.attrs = attr;
    c2.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&c2, attn_merge_kernel, a);
}

}  // namespace tfl
