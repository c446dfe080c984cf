// Seeded sampling of one token id per row from bf16 logits: the GPU draw the
// pages name beside argmax ("argmax or tf_sample_full", pull request #1415,
// section "How"), with temperature, top-k and top-p as in the release's
// recommended generation settings.  The pages fix no algorithm; the reading:
//   1. candidates: the ids whose logit is at least the k-th largest logit
//      (counted with multiplicity, ties included); all ids when k is 0 or >= V;
//   2. a logit value v weighs w(v) = exp((v - z_max) / T) (double); the mass of
//      a value is (candidates holding it) x w(v);
//   3. nucleus: walking the distinct candidate values from the largest down,
//      the first value at which the running mass reaches p x (candidates' mass)
//      is the cut; the nucleus is every candidate at or above it (all
//      candidates when p >= 1), its mass the running mass at the cut;
//   4. draw: with the caller's uniform u in [0, 1), the smallest id of the
//      nucleus whose running weight in id order exceeds u x (nucleus mass);
//      the largest nucleus id if rounding leaves none.
// A row holding NaN or +-Inf gets -1 and raises the non-finite status bit.
//
// Five launches; every sum is double, in a fixed order:
//   hist  (64 CTAs per row): CTA (i, c) reads the i-th 8th of the row and
//         counts, in shared memory, the finite logits whose order key (16 bits,
//         order-preserving, -0 folded into +0) is c mod 8, then adds its nonzero
//         counts to the row's counts; it raises the row's non-finite flag and
//         largest key;
//   range (64 CTAs per row): the weights of the keys that occur in a run of
//         1,024 keys, and the run's count and mass (count x weight);
//   cut   (one CTA per row): the top-k cut, the candidates' mass and the
//         nucleus cut, each by a walk over the 64 runs from the largest keys
//         down, then a scan inside the run where the walk crosses; the draw's
//         target u x (nucleus mass);
//   seg   (64 CTAs per row): zeroes the counts again (every call leaves them
//         zero; the model starts them zero), then the nucleus weight of each
//         64th of the ids;
//   draw  (one CTA per row): the 64th where the running weight passes the
//         target, then the id inside it.
// A scan over a CTA's threads goes through warp 0 (each lane sums a run of
// consecutive threads' partials in order, then a shuffle tree over the lanes),
// which keeps the double-precision work small; a crossing is claimed by the
// lowest thread whose running value passes the goal.  A row's result does not
// vary from run to run, and it differs from a plain sequential evaluation only
// when u x mass falls within rounding of a cumulative boundary.  Order keys
// 0..127 and 65,408..65,535 belong to the NaN and +-Inf patterns and never hold
// a count; their slots carry the row's parameters from one launch to the next.
#include "common.cuh"

namespace tfl {
namespace {

constexpr int kKeys = 65536;
constexpr int kKeyLo = 128, kKeyHi = 65407;  // order keys of finite bf16 values
constexpr int kRuns = 64, kRun = kKeys / kRuns;  // runs of 1,024 keys: range and cut CTAs, one key per thread
constexpr int kKeyThreads = kRun;
constexpr int kParts = 64;                       // 64ths of the ids: hist, seg and draw
constexpr int kIdThreads = 512;
// parameter slots (counts: unsigned, wtab: double) at keys that hold no finite value
constexpr int kPBad = 0, kPMax = 1, kPCut = 2, kPSkip = 3;  // counts: non-finite flag and largest key (raised by
                                                             // hist, cleared by cut), nucleus cut key, skip flag
constexpr int kPLast = 64;                                   // counts: last nucleus id per 64th
constexpr int kPRunC = kKeyHi + 1;                           // counts: count per run
constexpr int kPTarget = 0, kPSeg = 64, kPRunM = kKeyHi + 1; // wtab: draw target, nucleus weight per 64th, mass per run
static_assert(kPLast + kParts <= kKeyLo && kPSeg + kParts <= kKeyLo, "parameter slots below the finite keys");
static_assert(kPRunC + kRuns <= kKeys && kPRunM + kRuns <= kKeys, "parameter slots above the finite keys");

__device__ __forceinline__ uint32_t order_key(uint16_t b) {
    if (b == 0x8000u) b = 0;  // -0 and +0 are the same value
    return (b & 0x8000u) ? (uint32_t)(~b & 0xFFFFu) : (uint32_t)(b | 0x8000u);
}
__device__ __forceinline__ double key_value(uint32_t k) {
    const uint16_t b = (k & 0x8000u) ? (uint16_t)(k & 0x7FFFu) : (uint16_t)(~k & 0xFFFFu);
    return (double)__bfloat162float(__ushort_as_bfloat16(b));
}
__device__ __forceinline__ bool finite_key(int key) { return key >= kKeyLo && key <= kKeyHi; }

// Prefix of v over the NT threads in thread order: P(t) = v(0) + ... + v(t-1)
// as one running sum per group of NT/32 consecutive threads (warp 0, lane =
// group) started from a shuffle-tree scan of the group totals.  ex = P(t),
// in = P(t+1) (the next thread's ex; the last thread's is the total).
template <int NT>
__device__ __forceinline__ void scan_d(double v, double* sh, double& ex, double& in, double& total) {
    constexpr int G = NT / 32;
    const int tid = threadIdx.x, lane = tid & 31;
    sh[tid] = v;
    __syncthreads();
    if (tid < 32) {
        double g = 0.0;
#pragma unroll 4
        for (int i = 0; i < G; ++i) g += sh[lane * G + i];
        double x = g;  // inclusive over the groups
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x = y + x;
        }
        double run = __shfl_up_sync(0xffffffffu, x, 1);
        if (lane == 0) run = 0.0;
        for (int i = 0; i < G; ++i) {
            const double t = sh[lane * G + i];
            sh[lane * G + i] = run;
            run += t;
        }
        if (lane == 31) sh[NT] = x;
    }
    __syncthreads();
    total = sh[NT];
    ex = sh[tid];
    in = tid + 1 < NT ? sh[tid + 1] : total;
    __syncthreads();
}

// Total of v over the NT threads (the same association as scan_d's total).
template <int NT>
__device__ __forceinline__ double sum_d(double v, double* sh) {
    constexpr int G = NT / 32;
    const int tid = threadIdx.x, lane = tid & 31;
    sh[tid] = v;
    __syncthreads();
    if (tid < 32) {
        double g = 0.0;
#pragma unroll 4
        for (int i = 0; i < G; ++i) g += sh[lane * G + i];
        double x = g;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x = y + x;
        }
        if (lane == 31) sh[NT] = x;
    }
    __syncthreads();
    const double total = sh[NT];
    __syncthreads();
    return total;
}

// Inclusive and exclusive prefix of an integer over the block (exact).
__device__ __forceinline__ void scan_ll(long long v, long long* sh, long long& excl, long long& incl) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh[warp] = x;
    __syncthreads();
    if (warp == 0) {
        long long t = lane < nw ? sh[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        sh[32 + lane] = t;
    }
    __syncthreads();
    incl = (warp == 0 ? 0 : sh[32 + warp - 1]) + x;
    excl = incl - v;
    __syncthreads();
}

// Eight consecutive logits starting at id i (a multiple of 8) as raw bf16 bits;
// ids at or past V read as 0.  One 16-byte load when the row allows it.
__device__ __forceinline__ void load8(const uint16_t* z, int i, int V, bool vec, uint16_t (&b)[8]) {
    if (vec && i + 8 <= V) {
        const uint4 w = __ldg(reinterpret_cast<const uint4*>(z + i));
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            b[2 * e] = (uint16_t)(u[e] & 0xFFFFu);
            b[2 * e + 1] = (uint16_t)(u[e] >> 16);
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) b[e] = i + e < V ? z[i + e] : (uint16_t)0;
    }
}

// Ids of 64th `part` of a row: lo .. hi-1, lo a multiple of 8.
__device__ __forceinline__ void part_ids(int V, int part, int& lo, int& hi) {
    const int len = (V + 8 * kParts - 1) / (8 * kParts) * 8;
    lo = min(V, part * len);
    hi = min(V, lo + len);
}

// This thread's ids of 64th `part` (seg and draw split a 64th the same way):
// i0 .. i1-1, i0 a multiple of 8.
__device__ __forceinline__ void part_chunk(int V, int part, int& i0, int& i1) {
    int lo, hi;
    part_ids(V, part, lo, hi);
    const int chunk = (hi - lo + 8 * kIdThreads - 1) / (8 * kIdThreads) * 8;
    i0 = min(hi, lo + (int)threadIdx.x * chunk);
    i1 = min(hi, i0 + chunk);
}

// hist: CTA (8 i + c, row) counts the keys = c mod 8 among the ids of the i-th
// 8th of the row, then adds them to the counts (at most 8 additions per key).
constexpr int kHistParts = 8, kHistClasses = 8;
static_assert(kHistParts * kHistClasses == kParts, "hist grid");
__global__ void __launch_bounds__(kIdThreads) sample_hist_kernel(const bf16* logits, int V, unsigned* counts_all) {
    __shared__ unsigned hist[kKeys / kHistClasses];
    pdl_wait();
    pdl_trigger();
    const int ip = blockIdx.x / kHistClasses, kc = blockIdx.x % kHistClasses, row = blockIdx.y, tid = threadIdx.x;
    const uint16_t* z = reinterpret_cast<const uint16_t*>(logits) + (size_t)row * V;
    unsigned* counts = counts_all + (size_t)row * kKeys;
    const bool vec = ((reinterpret_cast<uintptr_t>(z) & 15u) == 0);
    for (int j = tid; j < kKeys / kHistClasses; j += kIdThreads) hist[j] = 0u;
    __syncthreads();
    const int len = (V + 8 * kHistParts - 1) / (8 * kHistParts) * 8;
    const int lo = min(V, ip * len), hi = min(V, lo + len);
    unsigned kmax = 0u;
    bool bad = false;
    for (int g0 = lo + 8 * tid; g0 < hi; g0 += 2 * 8 * kIdThreads) {
        uint16_t b[2][8];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int g = g0 + r * 8 * kIdThreads;
            if (g < hi) load8(z, g, V, vec, b[r]);
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int g = g0 + r * 8 * kIdThreads;
            if (g >= hi) continue;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if (g + e >= hi) continue;
                if ((b[r][e] & 0x7F80u) == 0x7F80u) {
                    bad = true;
                    continue;
                }
                const uint32_t k = order_key(b[r][e]);
                kmax = max(kmax, k);
                if ((int)(k % kHistClasses) == kc) atomicAdd(&hist[k / kHistClasses], 1u);
            }
        }
    }
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    bad = __any_sync(0xffffffffu, bad);
    if ((tid & 31) == 0) {
        if (kmax != 0u) atomicMax(&counts[kPMax], kmax);
        if (bad) atomicOr(&counts[kPBad], 1u);
    }
    __syncthreads();
    for (int j = tid; j < kKeys / kHistClasses; j += kIdThreads) {
        const unsigned c = hist[j];
        if (c != 0u) atomicAdd(&counts[j * kHistClasses + kc], c);
    }
}

// The key of this thread in run r (thread 0 holds the run's largest key).
__device__ __forceinline__ int run_key(int r) { return r * kRun + kRun - 1 - (int)threadIdx.x; }

// range: the weights exp((v - z_max) / T) of the keys that occur in run `part`
// (listed first, in any order: each weight is computed on its own, and the
// double-precision exponentials then run in full warps), and the run's count
// and mass (the cut launch trims the run holding the top-k cut).
__global__ void __launch_bounds__(kKeyThreads) sample_range_kernel(double temperature, unsigned* counts_all,
                                                                   double* wtab_all) {
    __shared__ double shd[kKeyThreads + 1], wsh[kRun];
    __shared__ uint16_t nz[kRun];
    __shared__ unsigned s_nz, s_c;
    pdl_wait();
    pdl_trigger();
    const int part = blockIdx.x, row = blockIdx.y, tid = threadIdx.x;
    unsigned* counts = counts_all + (size_t)row * kKeys;
    double* wtab = wtab_all + (size_t)row * kKeys;
    if (counts[kPBad] != 0u) return;
    if (tid == 0) {
        s_nz = 0u;
        s_c = 0u;
    }
    __syncthreads();
    const int key = run_key(part);
    const unsigned c = finite_key(key) ? counts[key] : 0u;
    if (c != 0u) nz[atomicAdd(&s_nz, 1u)] = (uint16_t)tid;
    const unsigned cw = __reduce_add_sync(0xffffffffu, c);
    if ((tid & 31) == 0) atomicAdd(&s_c, cw);
    __syncthreads();
    const double z_max = key_value(counts[kPMax]);
    for (int q = tid; q < (int)s_nz; q += kKeyThreads) {
        const int t = nz[q], k = run_key(part) + tid - t;  // key of thread t
        const double w = exp((key_value(k) - z_max) / temperature);
        wsh[t] = w;
        wtab[k] = w;
    }
    __syncthreads();
    const double m = sum_d<kKeyThreads>(c != 0u ? (double)c * wsh[tid] : 0.0, shd);
    if (tid == 0) {
        counts[kPRunC + part] = s_c;
        wtab[kPRunM + part] = m;
    }
}

// cut: top-k cut, candidates' mass, nucleus cut, target = u x nucleus mass.
__global__ void __launch_bounds__(kKeyThreads) sample_cut_kernel(int V, int top_k, double top_p, const float* u,
                                                                 int32_t* ids, int* status, unsigned* counts_all,
                                                                 double* wtab_all) {
    __shared__ double shd[kKeyThreads + 1], s_runm[kRuns];
    __shared__ long long shl[64];
    __shared__ unsigned s_cut_k, s_cut, s_runc[kRuns], s_bad;
    __shared__ int s_rk, s_rp, s_thr;
    __shared__ long long s_basec;
    __shared__ double s_basem, s_mass, s_total;
    pdl_wait();
    pdl_trigger();
    const int row = blockIdx.x, tid = threadIdx.x;
    unsigned* counts = counts_all + (size_t)row * kKeys;
    double* wtab = wtab_all + (size_t)row * kKeys;
    if (tid == 0) {  // the flags hist raised, passed on to seg and draw and cleared for the next call
        const unsigned bad = counts[kPBad];
        s_bad = bad;
        counts[kPSkip] = bad;
        counts[kPBad] = 0u;
        counts[kPMax] = 0u;
        if (bad != 0u) {
            ids[row] = -1;
            atomicOr(status, kStatusNonFinite);
        }
    }
    if (tid < kRuns) {
        s_runc[tid] = counts[kPRunC + tid];
        s_runm[tid] = wtab[kPRunM + tid];
    }
    __syncthreads();
    if (s_bad != 0u) return;
    // 1. the run holding the k-th largest value counted with multiplicity
    if (tid == 0) {
        int rk = -1;
        long long run = 0;
        if (top_k > 0 && top_k < V) {
            for (int r = kRuns - 1; r >= 0; --r) {
                const long long c = s_runc[r];
                if (run + c >= top_k) {
                    rk = r;
                    break;
                }
                run += c;
            }
        }
        s_rk = rk;
        s_basec = run;
        s_cut_k = 0u;  // all ids, unless the scan below sets a cut
        s_thr = kKeyThreads;
    }
    __syncthreads();
    const int rk = s_rk;
    // 2. the cut key inside that run (an exact integer scan: one claimant) and
    // the mass of the run's keys at or above it
    double partial = 0.0;
    if (rk >= 0) {
        const int key = run_key(rk);
        const unsigned c = finite_key(key) ? counts[key] : 0u;
        long long ex, in;
        scan_ll(c, shl, ex, in);
        const long long base = s_basec;
        if (base + ex < top_k && base + in >= top_k) s_cut_k = (unsigned)key;
        __syncthreads();
        const double w = c != 0u ? wtab[key] : 0.0;
        partial = sum_d<kKeyThreads>((c != 0u && (unsigned)key >= s_cut_k) ? (double)c * w : 0.0, shd);
    }
    const unsigned cut_k = s_cut_k;
    // 3. candidates' mass: the runs above the cut's run from the largest down,
    // then the trimmed run; the nucleus run: where that walk reaches p x mass
    auto run_mass = [&](int r) { return r > rk ? s_runm[r] : (r == rk ? partial : 0.0); };
    const int r_end = rk >= 0 ? rk : 0;
    if (tid == 0) {
        double total = 0.0;
        for (int r = kRuns - 1; r >= r_end; --r) total += run_mass(r);
        int rp = -1;
        double run = 0.0;
        if (top_p < 1.0) {
            const double goal = top_p * total;
            for (int r = kRuns - 1; r >= r_end; --r) {
                const double m = run_mass(r);
                if (run + m >= goal) {
                    rp = r;
                    break;
                }
                run += m;
            }
        }
        s_rp = rp;
        s_basem = run;
        s_total = total;
        s_cut = cut_k;
        s_mass = total;
    }
    __syncthreads();
    const int rp = s_rp;
    // 4. the nucleus cut inside that run: the key of the lowest thread whose
    // running mass reaches the goal; the nucleus mass is that running mass
    // (none claims only if rounding keeps the run below the goal: every candidate)
    if (rp >= 0) {
        const int key = run_key(rp);
        const unsigned c = finite_key(key) ? counts[key] : 0u;
        const double w = c != 0u ? wtab[key] : 0.0;
        double ex, in, tot;
        scan_d<kKeyThreads>((c != 0u && (unsigned)key >= cut_k) ? (double)c * w : 0.0, shd, ex, in, tot);
        const double base = s_basem, goal = top_p * s_total;
        const bool claim = c != 0u && (unsigned)key >= cut_k && base + in >= goal;
        if (claim) atomicMin(&s_thr, tid);
        __syncthreads();
        if (tid == s_thr) {
            s_cut = (unsigned)key;
            s_mass = base + in;
        }
    }
    __syncthreads();
    if (tid == 0) {
        counts[kPCut] = s_cut;
        wtab[kPTarget] = (double)u[row] * s_mass;
    }
}

// Eight ids from g (a multiple of 8): which are nucleus ids below i1 (bit e
// for id g + e) and their weights (0 for the others).  The weight gathers are
// independent, so they are in flight together.
__device__ __forceinline__ unsigned group8(const uint16_t* z, int V, bool vec, int g, int i1, unsigned cut,
                                           const double* wtab, double (&w)[8]) {
    uint16_t b[8];
    load8(z, g, V, vec, b);
    unsigned m = 0u;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const uint32_t k = order_key(b[e]);
        const bool in = g + e < i1 && k >= cut;
        w[e] = in ? wtab[k] : 0.0;
        m |= (in ? 1u : 0u) << e;
    }
    return m;
}

// Nucleus weight (sum in id order; a zero added for an id outside the nucleus
// leaves the sum unchanged) and last nucleus id of ids i0 .. i1-1.
__device__ __forceinline__ double chunk_weight(const uint16_t* z, int V, bool vec, int i0, int i1, unsigned cut,
                                               const double* wtab, int& last) {
    double s = 0.0;
    last = -1;
    for (int g = i0; g < i1; g += 8) {
        double w[8];
        const unsigned m = group8(z, V, vec, g, i1, cut, wtab, w);
#pragma unroll
        for (int e = 0; e < 8; ++e) s += w[e];
        if (m != 0u) last = g + 31 - __clz(m);
    }
    return s;
}

// seg: zero the counts again, then the nucleus weight and last nucleus id of
// each 64th of the ids.
__global__ void __launch_bounds__(kIdThreads) sample_seg_kernel(const bf16* logits, int V, unsigned* counts_all,
                                                                double* wtab_all) {
    __shared__ double shd[kIdThreads + 1];
    __shared__ int s_last;
    pdl_wait();
    pdl_trigger();
    const int part = blockIdx.x, row = blockIdx.y, tid = threadIdx.x;
    const uint16_t* z = reinterpret_cast<const uint16_t*>(logits) + (size_t)row * V;
    unsigned* counts = counts_all + (size_t)row * kKeys;
    double* wtab = wtab_all + (size_t)row * kKeys;
    {  // keys 1,024 part .. + 1,023 back to zero (cut, which read the counts last, has finished)
        const int k0 = part * (kKeys / kParts) + 2 * tid;
#pragma unroll
        for (int e = 0; e < 2; ++e)
            if (finite_key(k0 + e)) counts[k0 + e] = 0u;
    }
    if (counts[kPSkip] != 0u) return;
    const bool vec = ((reinterpret_cast<uintptr_t>(z) & 15u) == 0);
    const unsigned cut = counts[kPCut];
    if (tid == 0) s_last = -1;
    int i0, i1, last;
    part_chunk(V, part, i0, i1);
    const double total = sum_d<kIdThreads>(chunk_weight(z, V, vec, i0, i1, cut, wtab, last), shd);
    if (last >= 0) atomicMax(&s_last, last);
    __syncthreads();
    if (tid == 0) {
        wtab[kPSeg + part] = total;
        counts[kPLast + part] = (unsigned)s_last;
    }
}

// draw: the first 64th whose running weight passes the target, then the lowest
// thread there whose running weight passes it walks its ids.
__global__ void __launch_bounds__(kIdThreads) sample_draw_kernel(const bf16* logits, int V, int32_t* ids,
                                                                 unsigned* counts_all, double* wtab_all) {
    __shared__ double shd[kIdThreads + 1], s_segw[kParts];
    __shared__ int s_seg, s_thr, s_pick, s_segl[kParts];
    __shared__ double s_base;
    pdl_wait();
    pdl_trigger();
    const int row = blockIdx.x, tid = threadIdx.x;
    const uint16_t* z = reinterpret_cast<const uint16_t*>(logits) + (size_t)row * V;
    unsigned* counts = counts_all + (size_t)row * kKeys;
    double* wtab = wtab_all + (size_t)row * kKeys;
    if (counts[kPSkip] != 0u) return;
    const bool vec = ((reinterpret_cast<uintptr_t>(z) & 15u) == 0);
    const unsigned cut = counts[kPCut];
    const double target = wtab[kPTarget];
    if (tid < kParts) {
        s_segw[tid] = wtab[kPSeg + tid];
        s_segl[tid] = (int)counts[kPLast + tid];
    }
    __syncthreads();
    if (tid == 0) {
        double run = 0.0;
        int seg = -1, last = -1;
        for (int s = 0; s < kParts; ++s) {
            last = max(last, s_segl[s]);
            if (seg < 0) {
                const double nxt = run + s_segw[s];
                if (nxt > target) seg = s;
                else run = nxt;
            }
        }
        s_seg = seg;
        s_base = run;
        s_thr = kIdThreads;
        s_pick = seg < 0 ? last : s_segl[seg];  // rounding left no crossing: the last id
    }
    __syncthreads();
    const int seg = s_seg;
    if (seg >= 0) {
        int i0, i1, last;
        part_chunk(V, seg, i0, i1);
        double ex, in, total;
        scan_d<kIdThreads>(chunk_weight(z, V, vec, i0, i1, cut, wtab, last), shd, ex, in, total);
        const double base = s_base;
        if (last >= 0 && base + in > target) atomicMin(&s_thr, tid);
        __syncthreads();
        if (tid == s_thr) {
            double run = base + ex;
            int pick = -1;
            for (int g = i0; g < i1 && pick < 0; g += 8) {
                double w[8];
                const unsigned m = group8(z, V, vec, g, i1, cut, wtab, w);
                for (int e = 0; e < 8; ++e) {
                    if (!((m >> e) & 1u)) continue;
                    run += w[e];
                    if (run > target) {
                        pick = g + e;
                        break;
                    }
                }
            }
            s_pick = pick >= 0 ? pick : last;  // rounding kept the walk below the target: the chunk's last id
        }
    }
    __syncthreads();
    if (tid == 0) ids[row] = s_pick;
}

}  // namespace

cudaError_t launch_sample(const bf16* logits, int n_rows, int V, float temperature, int top_k, float top_p,
                          const float* u, int32_t* ids, int* status, unsigned* counts, double* wtab, cudaStream_t st,
                          bool pdl) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t c = {};
    c.stream = st;
    c.attrs = attr;
    c.numAttrs = pdl ? 1 : 0;
    c.blockDim = dim3(kIdThreads);
    c.gridDim = dim3(kParts, n_rows);
    cudaError_t e = cudaLaunchKernelEx(&c, sample_hist_kernel, logits, V, counts);
    if (e != cudaSuccess) return e;
    c.blockDim = dim3(kKeyThreads);
    c.gridDim = dim3(kRuns, n_rows);
    e = cudaLaunchKernelEx(&c, sample_range_kernel, (double)temperature, counts, wtab);
    if (e != cudaSuccess) return e;
    c.gridDim = dim3(n_rows);
    e = cudaLaunchKernelEx(&c, sample_cut_kernel, V, top_k, (double)top_p, u, ids, status, counts, wtab);
    if (e != cudaSuccess) return e;
    c.blockDim = dim3(kIdThreads);
    c.gridDim = dim3(kParts, n_rows);
    e = cudaLaunchKernelEx(&c, sample_seg_kernel, logits, V, counts, wtab);
    if (e != cudaSuccess) return e;
    c.gridDim = dim3(n_rows);
    return cudaLaunchKernelEx(&c, sample_draw_kernel, logits, V, ids, counts, wtab);
}

}  // namespace tfl
