// One decode step of one or two rows as a single persistent launch: the
// embedding, every decoder layer and the final norm + lm_head (the decode
// loop of pull request #1415, section "How", without a launch per operation).
//
// One CTA per SM (cooperative launch, so every CTA is resident), 384 threads:
// warp 11 is a TMA producer, warps 0..7 compute, warps 8..10 fold the
// attention units' warp partials handed to them by the compute warps.  The step is a fixed sequence
// of phases separated by grid barriers:
//   per layer: RMSNorm + QKV + RoPE + KV append | attention block partials |
//              merge | o + residual | RMSNorm + gate/up + SwiGLU | down + residual
//   then: final RMSNorm + lm_head.
// The producer walks the same sequence as the consumers and keeps a ring of
// eight 16 KB shared-memory stages full: the weight stages of the projections
// and the key/value tiles of the attention units (128 positions x 64 dims per
// stage, four stages per 128-key sub-block, up to four sub-blocks per unit of
// 512 keys) stream in while the consumers are still at a
// barrier, so each phase starts with data in place instead of paying a
// launch, a pipeline fill and a tail.  Only the key/value block holding this
// step's own rows waits for the barrier after the QKV phase.
//
// Every phase runs the arithmetic of the separate decode kernels (the shared
// device code of matvec_core.cuh and attn_core.cuh, the same work units and
// the same reduction orders), so a row's results are bit-identical to those
// of the multi-launch path: one-row steps here equal windows there.
//
// Grid barrier: thread 0 of each CTA fences, adds one to a counter and waits
// (acquire loads, bounded) until it reaches (barrier index) x (CTAs).  Every
// wait in the kernel is bounded; a timeout sets the device status and an abort
// flag that ends every other wait, and the kernel returns.
#include <cuda.h>

#include <algorithm>

#include "attn_core.cuh"
#include "common.cuh"
#include "matvec_core.cuh"
#include "tma.cuh"

namespace tfl {
namespace {

using mvc::kABytes;
using mvc::kConsumerWarps;
using mvc::kKbPerStage;

// warps 0-7 compute, then (steps whose attention units outnumber the CTAs)
// warps 8-10 combine attention partials, then the producer warp
constexpr int kCombineWarps = 3;
__host__ __device__ constexpr int producer_warp(bool combine) { return kConsumerWarps + (combine ? kCombineWarps : 0); }
__host__ __device__ constexpr int step_threads(bool combine) { return (producer_warp(combine) + 1) * 32; }
// Ring depth (stages) and activation space by rows.  (One row would leave room
// for 11 stages; measured, 8 stream as well or better.)
constexpr int kMaxDepth = 8;
__host__ __device__ constexpr int ring_depth(int) { return 8; }
__host__ __device__ constexpr int xs_bytes(int rows) { return rows * 22016 * 2; }  // down-projection lines
constexpr int kStage = kABytes;                       // 16 KB: one weight stage or one K/V tile
// the activation space also holds the attention's two query buffers and
// combine scratch, and the merge's scratch and staged partials
constexpr int kQBytes = attn::kPairs * kHeadDim * 2;  // one unit's queries
static_assert(2 * kQBytes + attn::comb_floats(attn::kGroupRows * 8) * 4 <= xs_bytes(kStepMaxRows),
              "attention scratch exceeds the activation space");
static_assert(2 * kQBytes + attn::comb_floats(8) * 4 <= xs_bytes(1), "one-row attention scratch");
static_assert(8192 + attn::kMergeStageFloats * 4 <= xs_bytes(1), "merge scratch exceeds the activation space");
constexpr int kRedBytes = kConsumerWarps * 4 * 32 * 4;
constexpr int kPhasesPerLayer = 6;
constexpr uint32_t kSpinLimit = 1u << 24;

enum Phase { PH_QKV, PH_ATTN, PH_MERGE, PH_O, PH_GATEUP, PH_DOWN, PH_HEAD };

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// The projection of a matvec phase, as the separate kernels describe it.
__device__ __forceinline__ MatvecArgs phase_args(const StepArgs& a, int l, int ph) {
    MatvecArgs e = {};
    e.n_rows = a.rows.n_rows;
    switch (ph) {
        case PH_QKV:
            e.mode = MV_QKV_ROPE;
            e.K = a.H;
            e.n_q = a.n_q;
            e.n_kv = a.n_kv;
            e.y = a.q;
            e.ldy = a.n_q * kHeadDim;
            e.cos_t = a.cos_t;
            e.sin_t = a.sin_t;
            e.layer = l;
            break;
        case PH_O:
            e.mode = MV_RESIDUAL;
            e.K = a.n_q * kHeadDim;
            e.n_out = a.H;
            e.h = a.h;
            break;
        case PH_GATEUP:
            e.mode = MV_SWIGLU;
            e.K = a.H;
            e.n_out = a.F;
            e.y = a.act;
            e.ldy = a.F;
            break;
        case PH_DOWN:
            e.mode = MV_RESIDUAL;
            e.K = a.F;
            e.n_out = a.H;
            e.h = a.h;
            break;
        default:  // PH_HEAD
            e.mode = MV_STORE;
            e.K = a.H;
            e.n_out = a.V;
            e.y = a.logits;
            e.ldy = a.V;
            break;
    }
    return e;
}

__device__ __forceinline__ const CUtensorMap* phase_maps(const StepArgs& a, int l, int ph) {
    switch (ph) {
        case PH_QKV: return a.wmaps + l * 7 + 0;
        case PH_O: return a.wmaps + l * 7 + 3;
        case PH_GATEUP: return a.wmaps + l * 7 + 4;
        case PH_DOWN: return a.wmaps + l * 7 + 6;
        default: return a.wmaps + a.layers * 7;
    }
}

__device__ __forceinline__ int phase_tiles(const MatvecArgs& e) {
    if (e.mode == MV_SWIGLU) return e.n_out / 8;
    if (e.mode == MV_QKV_ROPE) return (e.n_q + 2 * e.n_kv) * 8;
    return e.n_out / 16;
}

// Attention unit u of the step (the decode kernels' grid: 512-key unit, KV
// head, group of up to two rows of one stream); false when the unit lies past
// every row of its group.  nsub: its 128-key sub-blocks that any row sees.
// late: it reaches positions written this step.
struct Unit {
    int s, b, g, r0, nr, p_first, p_last, k0, nsub;
    bool late;
};
__device__ __forceinline__ bool attn_unit(const StepArgs& a, int u, int nunits, Unit& x) {
    x.b = u % nunits;
    const int rest = u / nunits;
    x.g = rest % a.n_kv;
    int z = rest / a.n_kv;
    bool found = false;
    for (int t = 0; t < a.rows.n_streams && !found; ++t) {
        const int rows = a.rows.row_start[t + 1] - a.rows.row_start[t];
        const int ng = (rows + attn::kGroupRows - 1) / attn::kGroupRows;
        if (z < ng) {
            x.s = t;
            x.r0 = a.rows.row_start[t] + z * attn::kGroupRows;
            x.nr = min(attn::kGroupRows, rows - z * attn::kGroupRows);
            found = true;
        } else {
            z -= ng;
        }
    }
    if (!found) return false;
    x.p_first = a.rows.pos0[x.s] + (x.r0 - a.rows.row_start[x.s]);
    x.p_last = x.p_first + x.nr - 1;
    x.k0 = x.b * kAttnUnit;
    if (x.k0 > x.p_last) return false;
    x.nsub = min(4, (x.p_last - x.k0) / kPage + 1);
    x.late = x.k0 + x.nsub * kPage > a.rows.pos0[x.s];
    return true;
}

__device__ __forceinline__ int attn_blocks(const StepArgs& a) {
    int max_pos = 0;
    for (int s = 0; s < a.rows.n_streams; ++s)
        max_pos = max(max_pos, a.rows.pos0[s] + a.rows.row_start[s + 1] - a.rows.row_start[s] - 1);
    return max_pos / kAttnUnit + 1;
}

__device__ __forceinline__ int attn_groups(const StepArgs& a) {
    int g = 0;
    for (int s = 0; s < a.rows.n_streams; ++s)
        g += (a.rows.row_start[s + 1] - a.rows.row_start[s] + attn::kGroupRows - 1) / attn::kGroupRows;
    return g;
}

// Waits until the grid barrier counter sync[0] reaches target; false on
// timeout or when another CTA has raised the abort flag sync[1].  One thread
// per CTA polls (acquire loads, no sleep: the wake-up follows the last arrival
// by one load); it gives up after `limit` polls or about a second of global
// time, whichever comes first.  A timeout sets kStatusDevice and raises the
// abort flag, which ends every other wait.
__device__ __forceinline__ bool wait_counter(unsigned* sync, int* status, unsigned target,
                                             uint32_t limit = kSpinLimit) {
    if (ld_acquire(sync) >= target) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 1; i < limit; ++i) {
        if (ld_acquire(sync) >= target) return true;
        if ((i & 63u) == 0u) {
            if (*((volatile unsigned*)sync + 1) != 0u) return false;
            if (global_ns() - t0 > kMbarWaitNs) break;
        }
    }
    atomicOr(status, kStatusDevice);
    atomicExch(sync + 1, 1u);
    return false;
}
__device__ __forceinline__ bool wait_counter(const StepArgs& a, unsigned target) {
    return wait_counter(a.sync, a.status, target);
}

struct ConsumerBar {
    __device__ __forceinline__ void operator()() const { named_barrier(1, kConsumerWarps * 32); }
};

struct RingPos {
    int stage;
    uint32_t phase;
    int depth;
    __device__ __forceinline__ void advance() {
        if (++stage == depth) {
            stage = 0;
            phase ^= 1u;
        }
    }
};

// ---- producer (the last warp, lane 0) -------------------------------------------
// Fills the ring in exactly the order the consumers drain it.
// rp / issued: the next ring stage and the number of stages armed so far
// (read by the caller to drain the ring after an abort).
__device__ void producer(const StepArgs& a, unsigned char* ring, uint64_t* full, uint64_t* empty,
                         volatile int* s_abort, RingPos& rp, long long& issued) {
    const uint64_t pol = policy_evict_first();
    const int G = gridDim.x;
    const int nblk = attn_blocks(a), units = nblk * a.n_kv * attn_groups(a);
    auto take = [&]() -> unsigned char* {
        if (*s_abort || !mbar_wait(&empty[rp.stage], rp.phase ^ 1u, a.status)) {
            *s_abort = 1;
            return nullptr;
        }
        mbar_arrive_expect_tx(&full[rp.stage], kStage);
        ++issued;  // the copy into this stage follows at once
        return ring + rp.stage * kStage;
    };
    auto weights = [&](int l, int ph) -> bool {
        const MatvecArgs e = phase_args(a, l, ph);
        const CUtensorMap* maps = phase_maps(a, l, ph);
        const int tiles = phase_tiles(e), nst = (e.K + 511) / 512;
        for (int t = blockIdx.x; t < tiles; t += G)
            for (int ks = 0; ks < nst; ++ks) {
                unsigned char* sA = take();
                if (!sA) return false;
                mvc::load_weights(e, maps, t, ks * kKbPerStage, sA, &full[rp.stage], pol);
                rp.advance();
            }
        return true;
    };
    for (int l = 0; l < a.layers; ++l) {
        if (!weights(l, PH_QKV)) return;
        // key/value tiles: blocks written by earlier steps first; the block(s)
        // holding this step's rows once every CTA has passed the QKV phase
        bool waited = false;
        for (int pass = 0; pass < 2; ++pass)
            for (int u = blockIdx.x; u < units; u += G) {
                Unit x;
                if (!attn_unit(a, u, nblk, x) || (int)x.late != pass) continue;
                if (x.late && !waited) {
                    if (!wait_counter(a, (unsigned)(l * kPhasesPerLayer + 1) * (unsigned)G)) {
                        *s_abort = 1;
                        return;
                    }
                    // the rows were written by generic stores of other CTAs; TMA reads through the async proxy
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    waited = true;
                }
                const KvView& kv = a.rows.kv[x.s];
                for (int j = 0; j < x.nsub; ++j) {
                    const int page = __ldg(kv.table + x.k0 / kPage + j);
                    for (int part = 0; part < 4; ++part) {  // K dims 0-63, K 64-127, V 0-63, V 64-127
                        unsigned char* dst = take();
                        if (!dst) return;
                        const int row0 = ((l * 2 + (part >> 1)) * kv.n_pages + page) * kPage;
                        tma_load_3d(dst, &a.kvmap[x.s], (part & 1) * 64, x.g, row0, &full[rp.stage], pol);
                        rp.advance();
                    }
                }
            }
        if (!weights(l, PH_O) || !weights(l, PH_GATEUP) || !weights(l, PH_DOWN)) return;
    }
    weights(0, PH_HEAD);
}

// ---- consumers (warps 0..7) ------------------------------------------------------
// Sub-block source over the ring (see attn::unit_partial): sub-block j of the
// unit is stages 4j .. 4j+3 after the unit's first (K lo, K hi, V lo, V hi),
// written by TMA with 128-byte swizzle (row r = a position, 64 dims).
struct RingSrc {
    unsigned char* ring;
    uint64_t* full;
    uint64_t* empty;
    RingPos base;
    int* status;
    volatile int* s_abort;
    int k0, p_last;
    // the four stages of the current sub-block (set by wait)
    int stage[4];
    uint32_t sa[4];
    __device__ __forceinline__ RingPos at(int i) const {
        RingPos r;
        r.stage = (base.stage + i) % base.depth;
        r.phase = base.phase ^ (uint32_t)(((base.stage + i) / base.depth) & 1);
        r.depth = base.depth;
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
            const RingPos r = at(4 * j + i);
            stage[i] = r.stage;
            sa[i] = smem_u32(ring + r.stage * kStage);
            if (!*s_abort && !mbar_wait(&full[r.stage], r.phase, status)) *s_abort = 1;
        }
        const int nv = min(kPage, p_last + 1 - (k0 + j * kPage));
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
    __device__ __forceinline__ void done(int) {
        __syncwarp();
        if ((threadIdx.x & 31) == 0)
            for (int i = 0; i < 4; ++i) mbar_arrive(&empty[stage[i]]);
    }
};

// Copies the queries of unit x's (row, head) pairs into the swizzled query
// buffer at q_u (pairs past the unit's are zero-filled), one 16-byte chunk per
// consumer thread, as an asynchronous copy group.
template <int GQ>
__device__ __forceinline__ void load_queries(const StepArgs& a, const Unit& x, uint32_t q_u) {
    static_assert(attn::kPairs * 16 == kConsumerWarps * 32, "one query chunk per consumer thread");
    const int p = threadIdx.x >> 4, c = threadIdx.x & 15, P = x.nr * GQ;
    const bf16* src = a.q;
    if (p < P) {
        const int row = x.r0 + p / GQ, head = x.g * GQ + p % GQ;
        src = a.q + (size_t)row * a.n_q * kHeadDim + (size_t)head * kHeadDim + c * 8;
    }
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(q_u + 2u * attn::swz(p, c * 8)), "l"(src),
                 "r"(p < P ? 16 : 0)
                 : "memory");
    wm::cp_async_commit();
}

// The partial of unit x with its queries already in the buffer at q_u.
// MAXNP: pair tiles the step's units can need (1 when every stream has one row).
// HANDOFF: the warps leave their partials in comb for the combine warps; pre()
// runs before they write into comb.
template <int GQ, int MAXNP, bool HANDOFF, class Pre>
__device__ __forceinline__ void attention_unit(const StepArgs& a, const AttnDecodeArgs& at, const Unit& x, uint32_t q_u,
                                               float* comb, unsigned char* ring, uint64_t* full, uint64_t* empty,
                                               RingPos rp, volatile int* s_abort, Pre pre) {
    const ConsumerBar bar;
    RingSrc src;
    src.ring = ring;
    src.full = full;
    src.empty = empty;
    src.base = rp;
    src.status = a.status;
    src.s_abort = s_abort;
    src.k0 = x.k0;
    src.p_last = x.p_last;
    attn::UnitGeom ug;
    ug.u = x.b;
    ug.g = x.g;
    ug.r0 = x.r0;
    ug.P = x.nr * GQ;
    ug.k0 = x.k0;
    ug.nsub = x.nsub;
    ug.p_first = x.p_first;
    ug.p_last = x.p_last;
    if (MAXNP == 1 || ug.P <= 8)
        attn::unit_partial_np<GQ, 1, HANDOFF>(at, ug, q_u, comb, src, bar, pre);
    else
        attn::unit_partial_np<GQ, MAXNP == 1 ? 1 : 2, HANDOFF>(at, ug, q_u, comb, src, bar, pre);
}

// This CTA's attention units in order: those reading only blocks written by
// earlier steps (pass 0), then those reaching this step's rows (pass 1).
struct UnitWalk {
    int pass, u;
    __device__ __forceinline__ bool next(const StepArgs& a, int nblk, int units, Unit& x) {
        for (;;) {
            u += gridDim.x;
            if (u >= units) {
                if (++pass == 2) return false;
                u = blockIdx.x;
            }
            if (u < units && attn_unit(a, u, nblk, x) && (int)x.late == pass) return true;
            if (u >= units) return false;
        }
    }
};

// The combine warps (96 threads): per layer, the partials of every attention
// unit of this CTA but its last (which the compute warps combine themselves),
// handed over through comb in the compute order; the same combine_pass
// arithmetic.  Every wait gives up once the abort flag rises; the three warps
// leave together.
template <int MAXNP>
__device__ void combiners(const StepArgs& a, float* comb, uint64_t* cfull, uint64_t* cempty, const int4* geom,
                          volatile int* s_abort) {
    const int ct = threadIdx.x - kConsumerWarps * 32;
    const int nblk = attn_blocks(a), units = nblk * a.n_kv * attn_groups(a);
    UnitWalk walk{0, (int)blockIdx.x - (int)gridDim.x};
    Unit x;
    int n = 0;
    while (walk.next(a, nblk, units, x)) ++n;
    const int handoffs = n > 0 ? n - 1 : 0;
    auto cbar = [] { named_barrier(2, kCombineWarps * 32); };
    const bool g7 = a.n_q / a.n_kv == 7;
    uint32_t use = 0;
    for (int l = 0; l < a.layers; ++l)
        for (int k = 0; k < handoffs; ++k) {
            const bool ok = mbar_wait_or_abort(cfull, use & 1u, s_abort, a.status);
            if (!named_barrier_and(2, kCombineWarps * 32, ok)) return;
            const int4 gm = *geom;
            constexpr int T = kCombineWarps * 32;
            if (MAXNP == 1 || gm.w <= 8) {
                if (g7)
                    attn::combine_pass<7, 8, T>(a.attn, gm.x, gm.y, gm.z, 0, gm.w, comb, ct, cbar);
                else
                    attn::combine_pass<8, 8, T>(a.attn, gm.x, gm.y, gm.z, 0, gm.w, comb, ct, cbar);
            } else {
                if (g7)
                    attn::combine_pass<7, 16, T>(a.attn, gm.x, gm.y, gm.z, 0, gm.w, comb, ct, cbar);
                else
                    attn::combine_pass<8, 16, T>(a.attn, gm.x, gm.y, gm.z, 0, gm.w, comb, ct, cbar);
            }
            cbar();  // every combine thread is done with comb
            if (ct == 0) mbar_arrive(cempty);
            ++use;
        }
}

template <int MAXNP, bool COMBINE>
__device__ void consumers(const StepArgs& a, unsigned char* ring, unsigned char* xs, float* red, float* red_norm,
                          uint64_t* full, uint64_t* empty, uint64_t* cfull, uint64_t* cempty, int4* geom,
                          volatile int* s_abort) {
    const int tid = threadIdx.x, lane = tid & 31, tig = lane & 3;
    const int R = a.rows.n_rows, G = gridDim.x;
    const int QD = a.n_q * kHeadDim, GQ = a.n_q / a.n_kv;
    const ConsumerBar bar;
    const uint32_t ring_u = smem_u32(ring), xs_u = smem_u32(xs);
    RingPos rp{0, 0u, ring_depth(a.rows.n_rows)};
    unsigned epoch = 0;
    uint32_t use = 0;  // hand-offs to the combine warps so far
    const int nblk = attn_blocks(a), units = nblk * a.n_kv * attn_groups(a);
    const AttnDecodeArgs& at = a.attn;

    unsigned long long* ts = a.ts ? a.ts + (size_t)blockIdx.x * step_ts_stride(a.layers) : nullptr;
    auto stamp = [&](int i) {
        if (ts && tid == 0) {
            unsigned long long t;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
            ts[i] = t;
        }
    };
    auto grid_barrier = [&]() -> bool {
        bar();  // this CTA's writes of the phase are done
        ++epoch;
        stamp(2 * epoch);
        if (tid == 0) {
            __threadfence();
            atomicAdd(a.sync, 1u);
            if (!wait_counter(a, epoch * (unsigned)G)) *s_abort = 1;
        }
        stamp(2 * epoch + 1);
        // every consumer thread takes the same decision (the producer may raise
        // the flag at any moment)
        return !named_barrier_or(1, kConsumerWarps * 32, *s_abort != 0);
    };
    auto matvec = [&](int l, int ph, auto row, const bf16* norm_w) {
        const MatvecArgs e = phase_args(a, l, ph);
        const int tiles = phase_tiles(e), nst = (e.K + 511) / 512, kblocks = e.K / 64;
        mvc::rows_to_lines(row, norm_w, a.eps, R, e.K, xs_u, red_norm, bar);
        for (int t = blockIdx.x; t < tiles; t += G)
            mvc::consume_tile<1>(e, a.rows, t, nst, R, ring_u, kStage, rp.depth, rp.stage, rp.phase, full, empty, red, s_abort,
                                 a.status, mvc::XFromLines{xs_u, R, kblocks, tig}, bar);
    };
    auto hrow = [&](int r) { return (const bf16*)a.h + (size_t)r * a.H; };
    auto aorow = [&](int r) { return (const bf16*)a.ao + (size_t)r * QD; };
    auto actrow = [&](int r) { return (const bf16*)a.act + (size_t)r * a.F; };
    auto erow = [&](int r) {
        const int id = a.ids[r];
        return (id >= 0 && id < a.V) ? a.embed + (size_t)id * a.H : a.zero_row;
    };

    stamp(0);
    for (int l = 0; l < a.layers; ++l) {
        // RMSNorm + QKV + RoPE + KV append
        if (l == 0) {
            // the residual stream starts as the embedding rows (zeros for an id out of range)
            if (blockIdx.x == 0) {
                for (int r = 0; r < R; ++r)
                    for (int i = tid * 8; i < a.H; i += kConsumerWarps * 32 * 8)
                        *reinterpret_cast<uint4*>(a.h + (size_t)r * a.H + i) =
                            *reinterpret_cast<const uint4*>(erow(r) + i);
                if (tid == 0)
                    for (int r = 0; r < R; ++r)
                        if (a.ids[r] < 0 || a.ids[r] >= a.V) atomicOr(a.status, kStatusBadToken);
            }
            matvec(0, PH_QKV, erow, a.norms[0]);
        } else {
            matvec(l, PH_QKV, hrow, a.norms[2 * l]);
        }
        if (!grid_barrier()) return;
        // attention block partials: blocks written by earlier steps, then this
        // step's; the next unit's queries are copied while this one runs; every
        // unit but the CTA's last hands its partials to the combine warps, the
        // last is combined here (once the combine warps are done with comb)
        {
            float* comb = reinterpret_cast<float*>(xs + 2 * kQBytes);
            UnitWalk walk{0, (int)blockIdx.x - G};
            Unit cur, nxt;
            bool have = walk.next(a, nblk, units, cur);
            int qb = 0;
            if (have) {
                if (GQ == 7) load_queries<7>(a, cur, xs_u); else load_queries<8>(a, cur, xs_u);
                wm::cp_async_wait_all();
            }
            while (have) {
                const bool have_next = walk.next(a, nblk, units, nxt);
                bar();  // the queries of cur are in place; the previous unit is done with the scratch
                const uint32_t q_cur = xs_u + qb * kQBytes, q_nxt = xs_u + (qb ^ 1) * kQBytes;
                if (have_next) {
                    if (GQ == 7) load_queries<7>(a, nxt, q_nxt); else load_queries<8>(a, nxt, q_nxt);
                }
                auto comb_free = [&] {
                    if (COMBINE && !*s_abort && !mbar_wait_or_abort(cempty, (use & 1u) ^ 1u, s_abort, a.status))
                        *s_abort = 1;
                };
                if (COMBINE && have_next) {
                    if (GQ == 7)
                        attention_unit<7, MAXNP, true>(a, at, cur, q_cur, comb, ring, full, empty, rp, s_abort,
                                                       comb_free);
                    else
                        attention_unit<8, MAXNP, true>(a, at, cur, q_cur, comb, ring, full, empty, rp, s_abort,
                                                       comb_free);
                    if (tid == 0) *geom = make_int4(cur.r0, cur.g, cur.b, cur.nr * GQ);
                    __syncwarp();
                    if ((tid & 31) == 0) mbar_arrive(cfull);
                    ++use;
                } else if (GQ == 7) {
                    attention_unit<7, MAXNP, false>(a, at, cur, q_cur, comb, ring, full, empty, rp, s_abort,
                                                    comb_free);
                } else {
                    attention_unit<8, MAXNP, false>(a, at, cur, q_cur, comb, ring, full, empty, rp, s_abort,
                                                    comb_free);
                }
                for (int j = 0; j < 4 * cur.nsub; ++j) rp.advance();
                wm::cp_async_wait_all();
                cur = nxt;
                have = have_next;
                qb ^= 1;
            }
        }
        if (!grid_barrier()) return;
        // merge: one (row, head) at a time
        {
            float* redm = reinterpret_cast<float*>(xs);
            float2* part = reinterpret_cast<float2*>(xs + 64);
            float* stage = reinterpret_cast<float*>(xs + 8192);
            for (int u = blockIdx.x; u < R * a.n_q; u += G)
                attn::merge<kConsumerWarps * 32>(at, u / a.n_q, u % a.n_q, tid, redm, part, bar, stage);
        }
        if (!grid_barrier()) return;
        matvec(l, PH_O, aorow, nullptr);
        if (!grid_barrier()) return;
        matvec(l, PH_GATEUP, hrow, a.norms[2 * l + 1]);
        if (!grid_barrier()) return;
        matvec(l, PH_DOWN, actrow, nullptr);
        if (!grid_barrier()) return;
    }
    matvec(0, PH_HEAD, hrow, a.final_norm);
    bar();
    stamp(1);
}

// MAXNP = 1: every stream of the step has one row (the attention's items have
// at most eight (row, head) pairs); 2: a stream has two rows.
// COMBINE: the variant with combine warps, for steps whose attention units
// outnumber the CTAs (each CTA then runs several units a layer).
template <int MAXNP, bool COMBINE>
__global__ void __launch_bounds__(step_threads(COMBINE), 1) step_kernel(const __grid_constant__ StepArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* ring =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int depth = ring_depth(a.rows.n_rows);
    unsigned char* xs = ring + depth * kStage;
    float* red = reinterpret_cast<float*>(xs + xs_bytes(a.rows.n_rows));
    float* red_norm = red + kRedBytes / 4;
    uint64_t* full = reinterpret_cast<uint64_t*>(red_norm + 8 * kStepMaxRows);
    uint64_t* empty = full + kMaxDepth;
    uint64_t* cfull = empty + kMaxDepth;  // comb holds a unit's warp partials
    uint64_t* cempty = cfull + 1;         // the combine warps are done with comb
    int4* geom = reinterpret_cast<int4*>(cempty + 1);  // the handed-over unit: (r0, g, unit, pairs)
    volatile int* s_abort = reinterpret_cast<volatile int*>(geom + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < depth; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        mbar_init(cfull, kConsumerWarps);
        mbar_init(cempty, 1);
        *s_abort = 0;
        mbar_init_fence();
    }
    __syncthreads();
    if (COMBINE && warp >= kConsumerWarps && warp < producer_warp(COMBINE)) {
        combiners<MAXNP>(a, reinterpret_cast<float*>(xs + 2 * kQBytes), cfull, cempty, geom, s_abort);
        return;
    }
    if (warp == producer_warp(COMBINE)) {
        if (lane == 0) {
            RingPos rp{0, 0u, depth};
            long long issued = 0;
            producer(a, ring, full, empty, s_abort, rp, issued);
            // after an abort, the copies already issued land before the CTA ends
            if (*s_abort) drain_ring(full, rp.depth, rp.stage, rp.phase, issued, a.status);
        }
        return;
    }
    consumers<MAXNP, COMBINE>(a, ring, xs, red, red_norm, full, empty, cfull, cempty, geom, s_abort);
}

// The two bounded waits of the step kernel run alone, each on something that
// never happens, so that their give-up path can be exercised: which = 0: the
// grid-barrier wait of thread 0 of every CTA on a counter target no CTA
// reaches (the first CTA to give up raises the abort flag, which ends the
// others' waits); which = 1: an mbarrier wait on a phase that never receives
// an arrival (no copy is issued to it).  Either way the status word gets
// kStatusDevice and the kernel returns.
__global__ void wait_probe_kernel(unsigned* sync, int* status, int which, uint32_t limit) {
    __shared__ uint64_t bar;
    if (which == 0) {
        if (threadIdx.x == 0) wait_counter(sync, status, 0xFFFFFFFFu, limit);
        return;
    }
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0u, status, limit);
    __syncthreads();
}

}  // namespace

cudaError_t launch_wait_probe(unsigned* sync, int* status, int which, uint32_t limit, int grid, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(sync, 0, 2 * sizeof(unsigned), st);
    if (e != cudaSuccess) return e;
    wait_probe_kernel<<<which == 0 ? grid : 1, 32, 0, st>>>(sync, status, which, limit);
    return cudaGetLastError();
}

int step_smem_bytes(int rows) {
    return 1024 + ring_depth(rows) * kStage + xs_bytes(rows) + kRedBytes + 8 * kStepMaxRows * 4 + 2 * kMaxDepth * 8 +
           2 * 8 + 16 + 64;
}

cudaError_t init_step_persistent() {
    const int smem = std::max(step_smem_bytes(1), step_smem_bytes(2));
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(step_kernel<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem))) return e;
    if ((e = cudaFuncSetAttribute(step_kernel<2, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem))) return e;
    if ((e = cudaFuncSetAttribute(step_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem))) return e;
    return cudaFuncSetAttribute(step_kernel<2, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

cudaError_t launch_step_persistent(const StepArgs& a, int grid, cudaStream_t st) {
    if (a.rows.n_rows < 1 || a.rows.n_rows > kStepMaxRows || a.rows.n_streams > kStepMaxRows || a.n_kv < 1 ||
        (a.n_q / a.n_kv != 7 && a.n_q / a.n_kv != 8) || a.n_q % a.n_kv != 0 || a.F > 22016)
        return cudaErrorInvalidValue;
    cudaError_t e = cudaMemsetAsync(a.sync, 0, 2 * sizeof(unsigned), st);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    // attention units of the step (as attn_blocks x n_kv x attn_groups)
    int max_pos = 0, groups = 0;
    for (int s = 0; s < a.rows.n_streams; ++s) {
        const int rows = a.rows.row_start[s + 1] - a.rows.row_start[s];
        max_pos = std::max(max_pos, a.rows.pos0[s] + rows - 1);
        groups += (rows + attn::kGroupRows - 1) / attn::kGroupRows;
    }
    const long long units = (long long)(max_pos / kAttnUnit + 1) * a.n_kv * groups;
    const bool combine = units > grid;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(step_threads(combine));
    cfg.dynamicSmemBytes = step_smem_bytes(a.rows.n_rows);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const bool one_row_streams = a.rows.n_rows == a.rows.n_streams;
    if (combine)
        return one_row_streams ? cudaLaunchKernelEx(&cfg, step_kernel<1, true>, a)
                               : cudaLaunchKernelEx(&cfg, step_kernel<2, true>, a);
    return one_row_streams ? cudaLaunchKernelEx(&cfg, step_kernel<1, false>, a)
                           : cudaLaunchKernelEx(&cfg, step_kernel<2, false>, a);
}

}  // namespace tfl
