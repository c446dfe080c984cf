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
// One CTA of 1,024 threads per row.  bf16 logits take at most 65,536 values:
// the CTA builds a count per value (order-preserving 16-bit keys, -0 folded
// into +0) in a per-row scratch, so the top-k cut is a count scan and every
// mass a sum over values in descending order; the draw is a scan over ids in
// contiguous chunks.  All scans run in a fixed order (per-thread chunks, then a
// shuffle tree), so a row's result does not vary from run to run.  Sums are
// double; an id differs from a plain sequential evaluation only when u x mass
// falls within rounding of a cumulative boundary.
#include "common.cuh"

namespace tfl {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kKeys = 65536;
constexpr int kKeysPerThread = kKeys / kThreads;  // 64, thread t owns keys descending from 65535 - 64 t

__device__ __forceinline__ uint32_t order_key(uint16_t b) {
    if (b == 0x8000u) b = 0;  // -0 and +0 are the same value
    return (b & 0x8000u) ? (uint32_t)(~b & 0xFFFFu) : (uint32_t)(b | 0x8000u);
}
__device__ __forceinline__ double key_value(uint32_t k) {
    const uint16_t b = (k & 0x8000u) ? (uint16_t)(k & 0x7FFFu) : (uint16_t)(~k & 0xFFFFu);
    return (double)__bfloat162float(__ushort_as_bfloat16(b));
}

// Inclusive and exclusive prefix of v over the block in thread order (fixed
// association: a shuffle tree inside each warp, then over the warp totals).
template <typename T>
__device__ __forceinline__ void block_scan(T v, T* sh, T& excl, T& incl, T& total) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    T x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const T y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x = y + x;
    }
    T ex_w = __shfl_up_sync(0xffffffffu, x, 1);
    if (lane == 0) ex_w = T(0);
    if (lane == 31) sh[warp] = x;
    __syncthreads();
    if (warp == 0) {
        T t = sh[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const T y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t = y + t;
        }
        sh[32 + lane] = t;  // inclusive over warps
    }
    __syncthreads();
    const T off = warp == 0 ? T(0) : sh[32 + warp - 1];
    excl = lane == 0 ? off : off + ex_w;
    incl = off + x;
    total = sh[32 + kWarps - 1];
    __syncthreads();
}

__global__ void __launch_bounds__(kThreads) sample_kernel(const bf16* logits, int V, double temperature, int top_k,
                                                          double top_p, const float* u, int32_t* ids, int* status,
                                                          unsigned* counts_all, double* wtab_all) {
    __shared__ double shd[64];
    __shared__ long long shl[64];
    __shared__ unsigned s_kmax;
    __shared__ int s_bad, s_pick, s_last;
    __shared__ unsigned s_cut_k, s_cut;
    __shared__ double s_mass;
    pdl_wait();
    pdl_trigger();
    const int row = blockIdx.x, tid = threadIdx.x;
    const uint16_t* z = reinterpret_cast<const uint16_t*>(logits) + (size_t)row * V;
    unsigned* counts = counts_all + (size_t)row * kKeys;
    double* wtab = wtab_all + (size_t)row * kKeys;

    // 1. counts per value, largest key, non-finite check
    for (int k = tid; k < kKeys; k += kThreads) counts[k] = 0u;
    if (tid == 0) {
        s_kmax = 0u;
        s_bad = 0;
        s_pick = -1;
        s_last = -1;
        s_cut_k = 0u;  // all ids, unless the top-k scan below sets a cut
    }
    __syncthreads();
    unsigned kmax = 0u;
    bool bad = false;
    for (int i = tid; i < V; i += kThreads) {
        const uint16_t b = z[i];
        if ((b & 0x7F80u) == 0x7F80u) {
            bad = true;
            continue;
        }
        const uint32_t k = order_key(b);
        atomicAdd(&counts[k], 1u);
        kmax = max(kmax, k);
    }
    if (bad) s_bad = 1;
    atomicMax(&s_kmax, kmax);
    __syncthreads();
    if (s_bad) {
        if (tid == 0) {
            ids[row] = -1;
            atomicOr(status, kStatusNonFinite);
        }
        return;
    }
    const double z_max = key_value(s_kmax);
    const int k_hi = kKeys - 1 - tid * kKeysPerThread;  // this thread's keys: k_hi down to k_hi - 63

    // 2. top-k cut (a key): the k-th largest value counted with multiplicity
    long long c_t = 0;
    for (int j = 0; j < kKeysPerThread; ++j) c_t += counts[k_hi - j];
    if (top_k > 0 && top_k < V) {
        long long ex, in, tot;
        block_scan<long long>(c_t, shl, ex, in, tot);
        if (ex < top_k && in >= top_k) {
            long long run = ex;
            for (int j = 0; j < kKeysPerThread; ++j) {
                run += counts[k_hi - j];
                if (run >= top_k) {
                    s_cut_k = (unsigned)(k_hi - j);
                    break;
                }
            }
        }
    }
    __syncthreads();
    const unsigned cut_k = s_cut_k;

    // 3. weights per value and the candidates' mass (values in descending order)
    double m_t = 0.0;
    for (int j = 0; j < kKeysPerThread; ++j) {
        const int key = k_hi - j;
        const unsigned c = counts[key];
        double w = 0.0;
        if (c != 0u && (unsigned)key >= cut_k) {
            w = exp((key_value(key) - z_max) / temperature);
            m_t += (double)c * w;
        }
        wtab[key] = w;
    }
    double ex, in, total;
    block_scan<double>(m_t, shd, ex, in, total);

    // 4. nucleus cut (default: every candidate, kept if rounding keeps the
    // crossing thread's own running sum below the goal)
    if (tid == 0) {
        s_cut = cut_k;
        s_mass = total;
    }
    __syncthreads();
    if (top_p < 1.0) {
        const double goal = top_p * total;
        if (ex < goal && in >= goal) {
            double run = ex;
            for (int j = 0; j < kKeysPerThread; ++j) {
                const int key = k_hi - j;
                const unsigned c = counts[key];
                if (c == 0u || (unsigned)key < cut_k) continue;
                run += (double)c * wtab[key];
                if (run >= goal) {
                    s_cut = (unsigned)key;
                    s_mass = run;
                    break;
                }
            }
        }
    }
    __syncthreads();
    const unsigned cut = s_cut;
    const double target = (double)u[row] * s_mass;

    // 5. draw over ids in contiguous chunks
    const int chunk = (V + kThreads - 1) / kThreads;
    const int i0 = tid * chunk, i1 = min(V, i0 + chunk);
    double s_t = 0.0;
    int last = -1;
    for (int i = i0; i < i1; ++i) {
        const uint32_t k = order_key(z[i]);
        if (k >= cut) {
            s_t += wtab[k];
            last = i;
        }
    }
    block_scan<double>(s_t, shd, ex, in, total);
    if (last >= 0) atomicMax(&s_last, last);
    if (ex <= target && in > target) {
        double run = ex;
        int pick = -1, lst = -1;
        for (int i = i0; i < i1; ++i) {
            const uint32_t k = order_key(z[i]);
            if (k < cut) continue;
            lst = i;
            run += wtab[k];
            if (run > target) {
                pick = i;
                break;
            }
        }
        s_pick = pick >= 0 ? pick : lst;
    }
    __syncthreads();
    if (tid == 0) ids[row] = s_pick >= 0 ? s_pick : s_last;
}

}  // namespace

cudaError_t launch_sample(const bf16* logits, int n_rows, int V, float temperature, int top_k, float top_p,
                          const float* u, int32_t* ids, int* status, unsigned* counts, double* wtab, cudaStream_t st,
                          bool pdl) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t c = {};
    c.gridDim = dim3(n_rows);
    c.blockDim = dim3(kThreads);
    c.stream = st;
    c.attrs = attr;
    c.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&c, sample_kernel, logits, V, (double)temperature, top_k, (double)top_p, u, ids, status,
                              counts, wtab);
}

}  // namespace tfl
