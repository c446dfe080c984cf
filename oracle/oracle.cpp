// Oracle: a plain, slow CPU forward of the bf16 GQA decoder (Llama family,
// Nanbeige4.3-33B shape), used ONLY as test infrastructure.
//
// Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
// leg may load this library.  It shares no code with the CUDA library under
// gqa_decoder_forward_gb300/csrc: no headers, no helpers, no tables.
//
// Arithmetic: every operation is carried out exactly (or in IEEE double, whose
// error is far below one bf16 step) and the result is rounded to bf16
// (round-to-nearest-even) only at the rounding points of HF modeling_llama run
// in bf16, as the Metal llama family pull request lists them
// ("A llama family on Metal ... pull request #1415", section "How"):
//   * residual add rounded:                h = bf16(h + f(h))
//   * RMSNorm:                             bf16(w * bf16(x * rsqrt(mean(x^2)+eps)))
//   * RoPE (NeoX half order):              bf16(bf16(x c) + bf16(o s)), o = rotate_half(x),
//                                          c, s = bf16 cos / sin of the fp32 angle
//   * SwiGLU:                              bf16(bf16(silu(g)) * u)
//   * projections:                         one sum, rounded once to bf16
// The float64-with-bf16-points design follows the same pull request's float64
// reference ("--bf16-points": each operation exact before the point).
//
// Readings where the pages are silent:
//   * attention: scores, softmax and P.V at full precision, output rounded once;
//     scale 1/sqrt(head_dim);
//   * inv_freq[i] = fl32(1 / fl32(theta^(2i/D))); angle = fl32(pos * inv_freq[i]);
//     cos/sin of that angle evaluated in double and rounded straight to bf16;
//   * silu(g) = g / (1 + exp(-g)) in double;
//   * argmax ties go to the lowest id; any non-finite logit in a row is an error.
//
// Every function is pinned by the tests against closed forms, brute force or
// library routines; the whole-model forward on random weights has no printed
// values to pin against and is pinned only through its components and
// invariants.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <cfenv>
#include <thread>
#include <vector>
#include <algorithm>
#include <functional>

namespace {

int g_threads = 0;  // 0 = std::thread::hardware_concurrency()
// Projection sums: 0 = in double (exact before the rounding point, the default
// reading); 1 = in fp32, one IEEE addition per term in increasing k order (the
// literal "fp32 sums rounded once" of the same pull request).  The second is a
// second faithful implementation of the method whose distance from the first
// measures how far two correct fp32-summing implementations may drift apart.
int g_fp32_sums = 0;

int thread_count() {
    if (g_threads > 0) return g_threads;
    unsigned n = std::thread::hardware_concurrency();
    return n == 0 ? 1 : (int)n;
}

// Runs body(i) for i in [0, n) split over the oracle's threads.  Each index is
// computed independently, so the split does not change any result.
void parallel_for(long n, const std::function<void(long)>& body) {
    int nt = thread_count();
    if (nt <= 1 || n < 2) {
        for (long i = 0; i < n; ++i) body(i);
        return;
    }
    if ((long)nt > n) nt = (int)n;
    std::vector<std::thread> pool;
    long chunk = (n + nt - 1) / nt;
    for (int t = 0; t < nt; ++t) {
        long lo = t * chunk, hi = std::min(n, lo + chunk);
        if (lo >= hi) break;
        pool.emplace_back([lo, hi, &body] { for (long i = lo; i < hi; ++i) body(i); });
    }
    for (auto& th : pool) th.join();
}

// ---- bf16 <-> double -------------------------------------------------------

double bf16_val(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return (double)f;
}

// Rounds a double to the nearest bf16 (8 significant bits, exponent range of
// fp32), ties to even; overflow goes to +-inf, NaN to the canonical quiet NaN.
uint16_t bf16_round(double x) {
    if (std::isnan(x)) return 0x7FC0;
    if (std::isinf(x)) return x > 0 ? 0x7F80 : 0xFF80;
    double r = 0.0;
    if (x != 0.0) {
        int e;
        std::frexp(x, &e);              // |x| = m * 2^e, 0.5 <= m < 1
        int q = e - 8;                  // weight of the last of 8 significant bits
        if (q < -133) q = -133;         // bf16 subnormal spacing is 2^-133
        double scaled = std::ldexp(x, -q);   // exact: a power-of-two scaling
        r = std::ldexp(std::nearbyint(scaled), q);  // current mode: nearest, ties to even
    } else {
        r = x;  // keeps the sign of zero
    }
    if (std::fabs(r) >= 0x1p128) return r > 0 ? 0x7F80 : 0xFF80;
    float f = (float)r;                 // exact: r has at most 8 significant bits
    uint32_t u;
    std::memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

float fl32(double x) { return (float)x; }  // IEEE round to nearest even

}  // namespace

extern "C" {

// ---- configuration ----------------------------------------------------------

void orc_set_threads(int n) { g_threads = n; }
int orc_get_threads(void) { return thread_count(); }
void orc_set_fp32_sums(int on) { g_fp32_sums = on ? 1 : 0; }
int orc_get_fp32_sums(void) { return g_fp32_sums; }

// ---- elementwise primitives ------------------------------------------------

uint16_t orc_bf16_from_double(double x) { return bf16_round(x); }
double orc_bf16_to_double(uint16_t b) { return bf16_val(b); }

void orc_bf16_round_array(const double* x, long n, uint16_t* out) {
    for (long i = 0; i < n; ++i) out[i] = bf16_round(x[i]);
}

// h = bf16(h + y), elementwise (the rounded residual add).
void orc_residual_add(uint16_t* h, const uint16_t* y, long n) {
    for (long i = 0; i < n; ++i) h[i] = bf16_round(bf16_val(h[i]) + bf16_val(y[i]));
}

// out = bf16(w * bf16(x * r)), r = 1 / sqrt(mean(x^2) + eps), per row of width H.
void orc_rmsnorm(const uint16_t* x, const uint16_t* w, int rows, int H, double eps, uint16_t* out) {
    for (int r = 0; r < rows; ++r) {
        const uint16_t* xr = x + (long)r * H;
        double ss = 0.0;
        for (int i = 0; i < H; ++i) { double v = bf16_val(xr[i]); ss += v * v; }
        double inv = 1.0 / std::sqrt(ss / H + eps);
        for (int i = 0; i < H; ++i) {
            double y = bf16_val(bf16_round(bf16_val(xr[i]) * inv));
            out[(long)r * H + i] = bf16_round(bf16_val(w[i]) * y);
        }
    }
}

// out[r][n] = bf16(sum_k W[n][k] * x[r][k]); W is [N][K] row-major (HF [out, in]).
// Each sum runs over k in increasing order, in double (default) or, with
// orc_set_fp32_sums(1), in fp32 (a product of two bf16 numbers is exact in
// fp32; each addition rounds to fp32).
void orc_linear(const uint16_t* W, int N, int K, const uint16_t* x, int rows, uint16_t* out) {
    std::vector<double> xd((size_t)rows * K);
    for (size_t i = 0; i < xd.size(); ++i) xd[i] = bf16_val(x[i]);
    const bool f32 = g_fp32_sums != 0;
    parallel_for(N, [&](long n) {
        const uint16_t* wn = W + n * (long)K;
        std::vector<double> wd(K);
        for (int k = 0; k < K; ++k) wd[k] = bf16_val(wn[k]);
        for (int r = 0; r < rows; ++r) {
            const double* xr = xd.data() + (size_t)r * K;
            if (f32) {
                float acc = 0.0f;
                for (int k = 0; k < K; ++k) acc = acc + (float)(wd[k] * xr[k]);
                out[(long)r * N + n] = bf16_round((double)acc);
            } else {
                double acc = 0.0;
                for (int k = 0; k < K; ++k) acc += wd[k] * xr[k];
                out[(long)r * N + n] = bf16_round(acc);
            }
        }
    });
}

// inv_freq[i] = fl32(1 / fl32(theta^(2i/D))), i = 0 .. D/2-1.
void orc_rope_inv_freq(double theta, int D, float* inv_freq) {
    for (int i = 0; i < D / 2; ++i) {
        float p = fl32(std::pow(theta, (2.0 * i) / D));
        inv_freq[i] = fl32(1.0 / (double)p);
    }
}

// cos/sin tables, [n_pos][D/2] bf16: c = bf16(cos(a)), s = bf16(sin(a)),
// a = fl32(pos * inv_freq[i]).
void orc_rope_table(double theta, int D, int n_pos, uint16_t* cos_out, uint16_t* sin_out) {
    std::vector<float> inv(D / 2);
    orc_rope_inv_freq(theta, D, inv.data());
    for (int p = 0; p < n_pos; ++p) {
        for (int i = 0; i < D / 2; ++i) {
            float a = fl32((double)(float)p * (double)inv[i]);
            cos_out[(long)p * (D / 2) + i] = bf16_round(std::cos((double)a));
            sin_out[(long)p * (D / 2) + i] = bf16_round(std::sin((double)a));
        }
    }
}

// NeoX rotation in place: x is [rows][nh][D]; row r sits at position pos[r].
// For j < D/2: out_j = bf16(bf16(x_j c_j) + bf16(-x_{j+D/2} s_j));
// for j >= D/2: out_j = bf16(bf16(x_j c_{j-D/2}) + bf16(x_{j-D/2} s_{j-D/2})).
void orc_rope_apply(uint16_t* x, int rows, int nh, int D, const int* pos,
                    const uint16_t* cos_t, const uint16_t* sin_t) {
    int half = D / 2;
    std::vector<double> v(D);
    for (int r = 0; r < rows; ++r) {
        for (int h = 0; h < nh; ++h) {
            uint16_t* xh = x + ((long)r * nh + h) * D;
            for (int j = 0; j < D; ++j) v[j] = bf16_val(xh[j]);
            const uint16_t* c = cos_t + (long)pos[r] * half;
            const uint16_t* s = sin_t + (long)pos[r] * half;
            for (int j = 0; j < D; ++j) {
                int i = j % half;
                double rot = j < half ? -v[j + half] : v[j - half];
                double a = bf16_val(bf16_round(v[j] * bf16_val(c[i])));
                double b = bf16_val(bf16_round(rot * bf16_val(s[i])));
                xh[j] = bf16_round(a + b);
            }
        }
    }
}

// Causal GQA attention.  q is [rows][NQ][D]; Kc, Vc are [n_pos][NKV][D];
// row r attends keys 0..pos[r]; q head h reads KV head h / (NQ/NKV).
// Scores, softmax and the weighted sum of V are exact up to double rounding;
// out [rows][NQ*D] is rounded once.
void orc_attention(const uint16_t* q, const int* pos, int rows, int NQ, int NKV, int D,
                   const uint16_t* Kc, const uint16_t* Vc, uint16_t* out) {
    int group = NQ / NKV;
    double scale = 1.0 / std::sqrt((double)D);
    parallel_for((long)rows * NQ, [&](long idx) {
        int r = (int)(idx / NQ), h = (int)(idx % NQ);
        int g = h / group;
        int n = pos[r] + 1;
        const uint16_t* qh = q + ((long)r * NQ + h) * D;
        std::vector<double> s(n);
        double mx = -INFINITY;
        for (int t = 0; t < n; ++t) {
            const uint16_t* kt = Kc + ((long)t * NKV + g) * D;
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += bf16_val(qh[d]) * bf16_val(kt[d]);
            s[t] = dot * scale;
            mx = std::max(mx, s[t]);
        }
        double l = 0.0;
        for (int t = 0; t < n; ++t) { s[t] = std::exp(s[t] - mx); l += s[t]; }
        for (int d = 0; d < D; ++d) {
            double acc = 0.0;
            for (int t = 0; t < n; ++t) acc += s[t] * bf16_val(Vc[((long)t * NKV + g) * D + d]);
            out[(long)r * NQ * D + (long)h * D + d] = bf16_round(acc / l);
        }
    });
}

// out = bf16(bf16(silu(g)) * u), silu(g) = g / (1 + exp(-g)).
void orc_swiglu(const uint16_t* g, const uint16_t* u, long n, uint16_t* out) {
    for (long i = 0; i < n; ++i) {
        double gv = bf16_val(g[i]);
        double sg = bf16_val(bf16_round(gv / (1.0 + std::exp(-gv))));
        out[i] = bf16_round(sg * bf16_val(u[i]));
    }
}

// Greedy id per row, ties to the lowest id.  Returns 0, or -1 if any logit in
// any row is NaN or +-Inf (that row's id is then set to -1).
int orc_argmax(const uint16_t* logits, int rows, int V, int32_t* ids) {
    int status = 0;
    for (int r = 0; r < rows; ++r) {
        const uint16_t* lr = logits + (long)r * V;
        int best = -1;
        double bv = 0.0;
        bool finite = true;
        for (int i = 0; i < V; ++i) {
            double v = bf16_val(lr[i]);
            if (!std::isfinite(v)) { finite = false; break; }
            if (best < 0 || v > bv) { best = i; bv = v; }
        }
        if (!finite) { ids[r] = -1; status = -1; } else { ids[r] = best; }
    }
    return status;
}

// Seeded sampling of one token per row (the GPU draw the pages name beside
// argmax: "argmax or tf_sample_full"; temperature, top-k and top-p as in the
// release's recommended settings).  The pages fix no algorithm; the reading
// over a row's bf16 logits z with T > 0, k >= 0,
// 0 < p, and a uniform u in [0, 1) given by the caller:
//   1. candidates C: all ids if k == 0 or k >= V, else the ids whose logit is at
//      least the k-th largest logit (counted with multiplicity; ties included);
//   2. weight of a logit value v: w(v) = exp((v - z_max) / T) in double;
//      mass of a value: (number of candidates holding it) * w(v);
//   3. nucleus N: walking the distinct candidate values from the largest down
//      and accumulating their mass, the first value at which the running mass
//      reaches p * (mass of C) is the cut; N = candidates with logit >= the cut
//      (all of C when p >= 1); W = the running mass at the cut;
//   4. draw: the smallest id j in N whose running sum of w over N in id order
//      exceeds u * W (the largest id of N if rounding leaves none).
// A row holding NaN or +-Inf gets -1 and the status -1.
int orc_sample(const uint16_t* logits, int rows, int V, double temperature, int top_k, double top_p,
               const double* u, int32_t* ids) {
    int status = 0;
    for (int r = 0; r < rows; ++r) {
        const uint16_t* lr = logits + (long)r * V;
        std::vector<double> z(V);
        bool finite = true;
        for (int i = 0; i < V; ++i) {
            z[i] = bf16_val(lr[i]);
            if (!std::isfinite(z[i])) finite = false;
        }
        if (!finite) {
            ids[r] = -1;
            status = -1;
            continue;
        }
        std::vector<double> sorted(z);
        std::sort(sorted.begin(), sorted.end(), std::greater<double>());
        const double z_max = sorted[0];
        const double kth = (top_k > 0 && top_k < V) ? sorted[top_k - 1] : sorted[V - 1];
        // distinct candidate values, largest first, with their counts
        std::vector<std::pair<double, long>> vals;
        for (double v : sorted) {
            if (v < kth) break;
            if (vals.empty() || vals.back().first != v) vals.push_back({v, 0});
            vals.back().second += 1;
        }
        auto w = [&](double v) { return std::exp((v - z_max) / temperature); };
        double total = 0.0;
        for (auto& vc : vals) total += (double)vc.second * w(vc.first);
        double cut = kth, mass = total;
        if (top_p < 1.0) {
            const double goal = top_p * total;
            double run = 0.0;
            for (auto& vc : vals) {
                run += (double)vc.second * w(vc.first);
                if (run >= goal) {
                    cut = vc.first;
                    mass = run;
                    break;
                }
            }
        }
        const double target = u[r] * mass;
        double run = 0.0;
        int pick = -1, last = -1;
        for (int i = 0; i < V; ++i) {
            if (z[i] < cut) continue;
            last = i;
            run += w(z[i]);
            if (run > target) {
                pick = i;
                break;
            }
        }
        ids[r] = pick >= 0 ? pick : last;
    }
    return status;
}

// ---- the model --------------------------------------------------------------

struct orc_config {
    int hidden, layers, n_q, n_kv, head_dim, ffn, vocab;
    double rope_theta;
    double rms_eps;
};

// Host pointers to bf16 tensors in HF layout; per-layer arrays have `layers` entries.
struct orc_weights {
    const uint16_t* embed;        // [vocab][hidden]
    const uint16_t* final_norm;   // [hidden]
    const uint16_t* lm_head;      // [vocab][hidden]
    const uint16_t* const* attn_norm;  // [hidden]
    const uint16_t* const* wq;    // [n_q*D][hidden]
    const uint16_t* const* wk;    // [n_kv*D][hidden]
    const uint16_t* const* wv;    // [n_kv*D][hidden]
    const uint16_t* const* wo;    // [hidden][n_q*D]
    const uint16_t* const* ffn_norm;   // [hidden]
    const uint16_t* const* wg;    // [ffn][hidden]
    const uint16_t* const* wu;    // [ffn][hidden]
    const uint16_t* const* wd;    // [hidden][ffn]
};

// One decoder layer over `rows` rows at positions pos[] (a window is causal:
// each row also sees the earlier rows of the same call).  h [rows][hidden] is
// updated in place; the rotated keys and the values of every row are written
// into this layer's cache Kc, Vc ([max_pos][n_kv][D]) before attention.
// cos_t/sin_t are tables built by orc_rope_table covering every pos[].
void orc_layer(const orc_config* c, int layer, const orc_weights* w,
               uint16_t* Kc, uint16_t* Vc, const int* pos, int rows, uint16_t* h,
               const uint16_t* cos_t, const uint16_t* sin_t) {
    const int H = c->hidden, D = c->head_dim, NQ = c->n_q, NKV = c->n_kv, F = c->ffn;
    std::vector<uint16_t> xn((size_t)rows * H), q((size_t)rows * NQ * D),
        k((size_t)rows * NKV * D), v((size_t)rows * NKV * D), o((size_t)rows * NQ * D),
        y((size_t)rows * H), g((size_t)rows * F), u((size_t)rows * F), a((size_t)rows * F);

    orc_rmsnorm(h, w->attn_norm[layer], rows, H, c->rms_eps, xn.data());
    orc_linear(w->wq[layer], NQ * D, H, xn.data(), rows, q.data());
    orc_linear(w->wk[layer], NKV * D, H, xn.data(), rows, k.data());
    orc_linear(w->wv[layer], NKV * D, H, xn.data(), rows, v.data());
    orc_rope_apply(q.data(), rows, NQ, D, pos, cos_t, sin_t);
    orc_rope_apply(k.data(), rows, NKV, D, pos, cos_t, sin_t);
    for (int r = 0; r < rows; ++r) {
        std::memcpy(Kc + (long)pos[r] * NKV * D, k.data() + (size_t)r * NKV * D, (size_t)NKV * D * 2);
        std::memcpy(Vc + (long)pos[r] * NKV * D, v.data() + (size_t)r * NKV * D, (size_t)NKV * D * 2);
    }
    orc_attention(q.data(), pos, rows, NQ, NKV, D, Kc, Vc, o.data());
    orc_linear(w->wo[layer], H, NQ * D, o.data(), rows, y.data());
    orc_residual_add(h, y.data(), (long)rows * H);

    orc_rmsnorm(h, w->ffn_norm[layer], rows, H, c->rms_eps, xn.data());
    orc_linear(w->wg[layer], F, H, xn.data(), rows, g.data());
    orc_linear(w->wu[layer], F, H, xn.data(), rows, u.data());
    orc_swiglu(g.data(), u.data(), (long)rows * F, a.data());
    orc_linear(w->wd[layer], H, F, a.data(), rows, y.data());
    orc_residual_add(h, y.data(), (long)rows * H);
}

// Final norm and lm_head: logits [rows][vocab] = bf16(Wlm . bf16 norm(h)).
void orc_head(const orc_config* c, const orc_weights* w, const uint16_t* h, int rows, uint16_t* logits) {
    std::vector<uint16_t> xn((size_t)rows * c->hidden);
    orc_rmsnorm(h, w->final_norm, rows, c->hidden, c->rms_eps, xn.data());
    orc_linear(w->lm_head, c->vocab, c->hidden, xn.data(), rows, logits);
}

// Full forward of `rows` token ids at positions pos[].  Kc/Vc are the caches
// of all layers, [layers][max_pos][n_kv][D].  hidden_trace (optional) receives
// the residual stream before layer 0 and after every layer:
// [layers+1][rows][hidden].  logits (optional) receives [rows][vocab].
// Returns 0, or -1 on a position outside [0, max_pos).
int orc_forward(const orc_config* c, const orc_weights* w, uint16_t* Kc, uint16_t* Vc, int max_pos,
                const int32_t* ids, const int* pos, int rows, uint16_t* logits, uint16_t* hidden_trace) {
    const int H = c->hidden, D = c->head_dim;
    int top = 0;
    for (int r = 0; r < rows; ++r) {
        if (pos[r] < 0 || pos[r] >= max_pos) return -1;
        top = std::max(top, pos[r] + 1);
    }
    std::vector<uint16_t> cos_t((size_t)top * (D / 2)), sin_t((size_t)top * (D / 2));
    orc_rope_table(c->rope_theta, D, top, cos_t.data(), sin_t.data());

    std::vector<uint16_t> h((size_t)rows * H);
    for (int r = 0; r < rows; ++r)
        std::memcpy(h.data() + (size_t)r * H, w->embed + (long)ids[r] * H, (size_t)H * 2);
    if (hidden_trace) std::memcpy(hidden_trace, h.data(), h.size() * 2);
    long layer_cache = (long)max_pos * c->n_kv * D;
    for (int l = 0; l < c->layers; ++l) {
        orc_layer(c, l, w, Kc + l * layer_cache, Vc + l * layer_cache, pos, rows, h.data(),
                  cos_t.data(), sin_t.data());
        if (hidden_trace) std::memcpy(hidden_trace + (size_t)(l + 1) * rows * H, h.data(), h.size() * 2);
    }
    if (logits) orc_head(c, w, h.data(), rows, logits);
    return 0;
}

}  // extern "C"
