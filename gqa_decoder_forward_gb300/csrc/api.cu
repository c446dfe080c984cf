// Host side of the C ABI declared in include/tfl.h: geometry qualification,
// workspace layout, paged KV objects, the RoPE table, and the launch sequence
// of a decode step and of a prompt chunk.  Everything that computes runs in
// the CUDA kernels of this directory; this file only validates and enqueues.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <algorithm>
#include <vector>

#include <cudaTypedefs.h>

#include "attn_decode.cuh"
#include "common.cuh"
#include "../../include/tfl.h"

using namespace tfl;

namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

int ok() {
    g_err.clear();
    return TFL_OK;
}

#define CK(call)                                                                                 \
    do {                                                                                         \
        cudaError_t e_ = (call);                                                                 \
        if (e_ != cudaSuccess)                                                                   \
            return fail(TFL_E_CUDA, "%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), __FILE__, __LINE__); \
    } while (0)

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Qualified geometries: the 33B shape (any 1..52-layer truncation of its stack)
// and the tiny test model (1..2 layers).
struct Geometry {
    const char* name;
    int hidden, max_layers, n_q, n_kv, head_dim, ffn, vocab;
    double theta;
};
const Geometry kQualified[] = {
    {"Nanbeige4.3-33B", 7168, 52, 56, 8, 128, 22016, 166912, 1.2e8},
    {"tiny test llama", 1024, 2, 8, 1, 128, 2816, 4096, 1.2e8},
};

const Geometry* qualified(const tfl_config* c) {
    for (const Geometry& g : kQualified)
        if (c->hidden == g.hidden && c->n_q == g.n_q && c->n_kv == g.n_kv && c->head_dim == g.head_dim &&
            c->ffn == g.ffn && c->vocab == g.vocab && c->rope_theta == g.theta && c->layers >= 1 &&
            c->layers <= g.max_layers)
            return &g;
    return nullptr;
}

int qualify(const tfl_config* c) {
    if (!c) return fail(TFL_E_ARG, "config is NULL");
    if (c->head_dim != kHeadDim)
        return fail(TFL_E_GEOMETRY, "head_dim %d refused: only heads of 128 are served", c->head_dim);
    if (!(c->rms_eps > 0.f) || !std::isfinite(c->rms_eps)) return fail(TFL_E_ARG, "rms_eps must be finite and > 0");
    if (!qualified(c))
        return fail(TFL_E_GEOMETRY,
                    "geometry refused: hidden %d, layers %d, %d q / %d kv heads of %d, ffn %d, vocab %d, theta %g is "
                    "not a qualified geometry (Nanbeige4.3-33B with 1..52 layers, or the tiny test llama)",
                    c->hidden, c->layers, c->n_q, c->n_kv, c->head_dim, c->ffn, c->vocab, c->rope_theta);
    if (c->max_rows < 1 || c->max_rows > kMaxChunkRows)
        return fail(TFL_E_ARG, "max_rows %d outside 1..%d", c->max_rows, kMaxChunkRows);
    if (c->max_decode_rows < 1 || c->max_decode_rows > kMaxDecodeRows)
        return fail(TFL_E_ARG, "max_decode_rows %d outside 1..%d", c->max_decode_rows, kMaxDecodeRows);
    if (c->max_context < 1 || c->max_context > (1 << 20))
        return fail(TFL_E_ARG, "max_context %d outside 1..%d", c->max_context, 1 << 20);
    return ok();
}

// Workspace layout (byte offsets, 256-byte aligned regions).
struct Layout {
    size_t h, xn, q, ao, act, pm, pl, po, cos_t, sin_t, status, wmaps, norms, sync, zero, ts, scounts, swtab, total;
    int max_blocks;
};


Layout layout(const tfl_config* c) {
    Layout L;
    const size_t rows = (size_t)std::max(c->max_rows, c->max_decode_rows);
    const size_t dr = (size_t)c->max_decode_rows;
    L.max_blocks = (c->max_context + kAttnUnit - 1) / kAttnUnit;  // decode-attention units per row
    const size_t qd = (size_t)c->n_q * kHeadDim;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = round_up(off + bytes, 256);
        return o;
    };
    L.h = take(rows * c->hidden * 2);
    L.xn = take(rows * std::max((size_t)c->hidden, qd) * 2);
    L.q = take(rows * qd * 2);
    L.ao = take(rows * qd * 2);
    L.act = take(rows * (size_t)c->ffn * 2);
    L.pm = take(dr * c->n_q * L.max_blocks * 4);
    L.pl = take(dr * c->n_q * L.max_blocks * 4);
    L.po = take(dr * c->n_q * L.max_blocks * (size_t)kHeadDim * 4);
    L.cos_t = take((size_t)c->max_context * 64 * 2);
    L.sin_t = take((size_t)c->max_context * 64 * 2);
    L.status = take(256);
    // the decode-step kernel's tables: every projection's TMA descriptor, the
    // norm weight pointers, the grid barrier words and a zero row
    L.wmaps = take(((size_t)c->layers * 7 + 1) * sizeof(CUtensorMap));
    L.norms = take((size_t)c->layers * 2 * sizeof(void*));
    L.sync = take(256);
    L.zero = take((size_t)c->hidden * 2);
    L.ts = take((size_t)kStepTsCtas * step_ts_stride(c->layers) * 8);
    // sampling scratch: a count and a weight per bf16 value, per row
    L.scounts = take(dr * 65536 * 4);
    L.swtab = take(dr * 65536 * 8);
    L.total = off;
    return L;
}

// Round a double to the nearest bf16 (ties to even) by rounding the double's
// 52-bit fraction at bit 45; valid for normal bf16 magnitudes, which is every
// nonzero cos/sin value of an fp32 angle.
uint16_t host_bf16(double x) {
    if (x == 0.0) return std::signbit(x) ? 0x8000 : 0;
    uint64_t u;
    std::memcpy(&u, &x, 8);
    const uint64_t lsb = (u >> 45) & 1u;
    u += (1ull << 44) - 1 + lsb;
    u &= ~((1ull << 45) - 1);
    double r;
    std::memcpy(&r, &u, 8);
    float f = (float)r;  // exact: 8 significant bits
    uint32_t b;
    std::memcpy(&b, &f, 4);
    return (uint16_t)(b >> 16);
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// A 3-D bf16 tensor map over a row-major [rows][K] matrix viewed as (64
// columns, rows, K/64 k-blocks) -- strides K*2 and 128 bytes -- with 128-byte
// swizzle and boxes of (64, box_rows, 8).
bool encode_map(CUtensorMap* m, const void* ptr, uint64_t K, uint64_t rows, uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn || ((uintptr_t)ptr & 15u) || K % 64 != 0 || box_rows < 1 || box_rows > 256) return false;
    cuuint64_t dims[3] = {64, rows, K / 64};
    cuuint64_t strides[2] = {K * 2, 128};
    cuuint32_t box[3] = {64, box_rows, 8};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// A 2-D bf16 tensor map over a row-major [rows][K] matrix with 128-byte
// swizzle and boxes of (64 columns, box_rows rows): the GEMM operands.
bool encode_map2d(CUtensorMap* m, const void* ptr, uint64_t K, uint64_t rows, uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn || ((uintptr_t)ptr & 15u) || K % 64 != 0 || box_rows < 1 || box_rows > 256) return false;
    cuuint64_t dims[2] = {K, rows};
    cuuint64_t strides[1] = {K * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// A 3-D bf16 tensor map over a KV cache's pages, viewed as rows of n_kv x 128
// (a row = one position of one (layer, K or V) page), boxes of 128 rows x one
// head x 64 dims with 128-byte swizzle: the key or value tile of one block.
bool encode_kv_map(CUtensorMap* m, const void* pages, int n_kv, uint64_t rows) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn || ((uintptr_t)pages & 15u)) return false;
    cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)n_kv, rows};
    cuuint64_t strides[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)n_kv * kHeadDim * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)kPage};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pages), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Index of the activation-row box for a call of `rows` rows: 1..8 -> 0..7,
// 16 -> 8, 32 -> 9, 64 -> 10.
int xbox_index(int rows) {
    const int xr = matvec_tma_x_rows(rows);
    return xr <= 8 ? xr - 1 : xr == 16 ? 8 : xr == 32 ? 9 : 10;
}
constexpr int kXBoxes = 11;

// Row counts up to which the projections after a norm apply the norm themselves.
constexpr int kMaxFusedNormRows = 8;

}  // namespace

// ---- model / kv objects --------------------------------------------------------

// Kernel families timed by tfl_profile (names in tfl_profile_kind).
enum Kind {
    K_EMBED, K_NORM, K_QKV, K_ATTN, K_MERGE, K_O, K_GATEUP, K_DOWN, K_LMHEAD, K_ARGMAX,
    K_GQKV, K_GO, K_GGATEUP, K_GDOWN, K_PATTN, K_STEP, K_SAMPLE, K_COUNT
};
const char* const kKindName[K_COUNT] = {"embed_rmsnorm", "rmsnorm", "matvec_qkv_rope", "attn_decode_block",
                                        "attn_decode_merge", "matvec_o_residual", "matvec_gate_up_swiglu",
                                        "matvec_down_residual", "matvec_lm_head", "argmax",
                                        "gemm_qkv_rope", "gemm_o_residual", "gemm_gate_up_swiglu",
                                        "gemm_down_residual", "attn_prefill", "decode_step_persistent",
                                        "sample"};

struct Mark {
    int kind;
    cudaEvent_t a, b;
};

struct tfl_model {
    tfl_config cfg;
    const bf16 *embed, *final_norm, *lm_head;
    std::vector<const bf16*> attn_norm, wq, wk, wv, wo, ffn_norm, wg, wu, wd;
    char* ws;
    Layout L;
    bf16 *h, *xn, *q, *ao, *act, *cos_t, *sin_t;
    float *pm, *pl, *po;
    int* status;
    CUtensorMap* d_wmaps;   // workspace copy of the decode matvec descriptors
    const bf16** d_norms;   // workspace copy of the norm weight pointers
    unsigned* sync;
    bf16* zero_row;
    unsigned long long* ts;  // decode-step phase stamps (written while profiling)
    unsigned* scounts;       // sampling scratch
    double* swtab;
    bool ts_valid = false;
    bool persistent = true; // decode steps of <= kStepMaxRows rows as one launch
    bool pdl;
    // TMA descriptors of every projection and of the activation buffers
    struct LayerMaps {
        CUtensorMap q, k, v, o, g, u, d;                // decode matvec (3-D)
        CUtensorMap gq, gk, gv, go, gg, gu, gd;         // prompt GEMM (2-D)
    };
    std::vector<LayerMaps> wmaps;
    CUtensorMap lm_map;
    CUtensorMap xmap_xn[kXBoxes], xmap_ao[kXBoxes], xmap_act[kXBoxes];  // by xbox_index(rows)
    CUtensorMap amap_xn, amap_ao, amap_act;  // GEMM activation operands (128-row boxes)
    int grid = 0;
    bool prof = false;
    std::vector<Mark> marks;         // recorded while profiling
    std::vector<cudaEvent_t> spare;  // event pool
    ~tfl_model() {
        for (Mark& k : marks) { cudaEventDestroy(k.a); cudaEventDestroy(k.b); }
        for (cudaEvent_t e : spare) cudaEventDestroy(e);
    }
};

namespace {

cudaEvent_t take_event(tfl_model* m) {
    if (!m->spare.empty()) {
        cudaEvent_t e = m->spare.back();
        m->spare.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

}  // namespace

// Launches `call`; while profiling, brackets it with CUDA events on stream st.
#define LAUNCH(m, kind, st, call)                                                 \
    do {                                                                          \
        cudaEvent_t a_ = nullptr, b_ = nullptr;                                   \
        if ((m)->prof) {                                                          \
            a_ = take_event(m);                                                   \
            b_ = take_event(m);                                                   \
            if (a_ && b_) CK(cudaEventRecord(a_, st));                            \
        }                                                                         \
        CK(call);                                                                 \
        if (a_ && b_) {                                                           \
            CK(cudaEventRecord(b_, st));                                          \
            (m)->marks.push_back(Mark{kind, a_, b_});                             \
        }                                                                         \
    } while (0)

struct tfl_kv {
    tfl_model* model;
    char* buf;
    int max_pos;
    int n_pages;
    int length;
    int* table;
    bf16* pages;
    CUtensorMap kvmap;  // 3-D over the pages: (128 dims, n_kv heads, rows), boxes of 128 rows x 64 dims
};

namespace {

size_t kv_table_bytes(int n_pages) { return round_up((size_t)n_pages * 4, 256); }

KvView view(const tfl_kv* kv) {
    KvView v;
    v.pages = kv->pages;
    v.table = kv->table;
    v.n_pages = kv->n_pages;
    v.pad_ = 0;
    return v;
}

// Launches the TMA matvec with weight maps w0..w2 and activation map xm (whose
// box rows must be matvec_tma_x_rows(e.n_rows)).
cudaError_t mv_launch(tfl_model* m, const MatvecArgs& e, const CUtensorMap* w0, const CUtensorMap* w1,
                      const CUtensorMap* w2, const CUtensorMap* xm, cudaStream_t st, bool pdl,
                      const bf16* norm_w = nullptr) {
    MatvecTmaArgs a;
    std::memset(&a, 0, sizeof a);
    if (norm_w) {  // e.x is the residual stream; the kernel applies the RMSNorm itself
        a.norm_w = norm_w;
        a.eps = m->cfg.rms_eps;
        a.depth = matvec_norm_depth(e.n_rows, e.K);
    }
    a.e = e;
    a.wmap[0] = *w0;
    if (w1) a.wmap[1] = *w1;
    if (w2) a.wmap[2] = *w2;
    a.xmap = *xm;
    a.x_rows_box = matvec_tma_x_rows(e.n_rows);
    a.tiles = matvec_tma_tiles(e);
    a.kstages = (e.K + 511) / 512;
    a.status = m->status;
    return launch_matvec_tma(a, m->grid, st, pdl);
}

// Decode attention partials: the TMA-fed kernel when every stream has one row
// (one (row, head) tile per item: its consumers keep up with the ring), the
// cp.async kernel otherwise (two-row items need the registers the producer
// warp would take).  Both give the same bits.
cudaError_t launch_attn_decode(const tfl_model* m, const AttnDecodeArgs& at, const KvMaps& maps, cudaStream_t st,
                               bool pdl) {
    bool one_row = true;
    for (int s = 0; s < at.rows.n_streams; ++s) one_row = one_row && at.rows.row_start[s + 1] - at.rows.row_start[s] == 1;
    return one_row ? launch_attn_block_tma(at, maps, m->status, m->grid, st, pdl) : launch_attn_block(at, st, pdl);
}

// The layer stack over n rows described by rm (decode kernels).  Input: ids
// (embedding gather) or h_in; output: the residual stream in m->h.
int run_layers(tfl_model* m, const RowMap& rm, const KvMaps& maps, const int32_t* ids, const void* h_in,
               cudaStream_t st) {
    const tfl_config& c = m->cfg;
    const int n = rm.n_rows, H = c.hidden, qd = c.n_q * kHeadDim;
    const bool pdl = m->pdl && st != nullptr;  // no programmatic launch on the legacy stream
    if (ids) {
        LAUNCH(m, K_EMBED, st,
               launch_embed_rmsnorm(ids, m->embed, c.vocab, m->attn_norm[0], c.rms_eps, n, H, m->h, m->xn, m->status,
                                    st, pdl));
    } else {
        CK(cudaMemcpyAsync(m->h, h_in, (size_t)n * H * 2, cudaMemcpyDeviceToDevice, st));
        LAUNCH(m, K_NORM, st, launch_rmsnorm(m->h, m->attn_norm[0], c.rms_eps, n, H, m->xn, st, false));
    }
    // up to 8 rows: each projection that follows a norm applies the norm itself
    const bool fuse = n <= kMaxFusedNormRows;
    for (int l = 0; l < c.layers; ++l) {
        if (l > 0 && !fuse)
            LAUNCH(m, K_NORM, st, launch_rmsnorm(m->h, m->attn_norm[l], c.rms_eps, n, H, m->xn, st, pdl));
        MatvecArgs a = {};
        a.mode = MV_QKV_ROPE;
        a.K = H;
        a.n_rows = n;
        a.x = m->xn;
        a.w0 = m->wq[l];
        a.w1 = m->wk[l];
        a.w2 = m->wv[l];
        a.n_q = c.n_q;
        a.n_kv = c.n_kv;
        a.y = m->q;
        a.ldy = qd;
        a.cos_t = m->cos_t;
        a.sin_t = m->sin_t;
        a.layer = l;
        a.rows = rm;
        const int xi = xbox_index(n);
        const tfl_model::LayerMaps& wm = m->wmaps[l];
        if (fuse) a.x = m->h;
        LAUNCH(m, K_QKV, st,
               mv_launch(m, a, &wm.q, &wm.k, &wm.v, &m->xmap_xn[xi], st, pdl, fuse ? m->attn_norm[l] : nullptr));

        AttnDecodeArgs at = {};
        at.q = m->q;
        at.out = m->ao;
        at.pm = m->pm;
        at.pl = m->pl;
        at.po = m->po;
        at.max_blocks = m->L.max_blocks;
        at.n_q = c.n_q;
        at.n_kv = c.n_kv;
        at.layer = l;
        at.rows = rm;
        LAUNCH(m, K_ATTN, st, launch_attn_decode(m, at, maps, st, pdl));
        LAUNCH(m, K_MERGE, st, launch_attn_merge(at, st, pdl));

        MatvecArgs o = {};
        o.mode = MV_RESIDUAL;
        o.K = qd;
        o.n_rows = n;
        o.x = m->ao;
        o.w0 = m->wo[l];
        o.n_out = H;
        o.h = m->h;
        LAUNCH(m, K_O, st, mv_launch(m, o, &wm.o, nullptr, nullptr, &m->xmap_ao[xi], st, pdl));

        if (!fuse) LAUNCH(m, K_NORM, st, launch_rmsnorm(m->h, m->ffn_norm[l], c.rms_eps, n, H, m->xn, st, pdl));

        MatvecArgs gu = {};
        gu.mode = MV_SWIGLU;
        gu.K = H;
        gu.n_rows = n;
        gu.x = m->xn;
        gu.w0 = m->wg[l];
        gu.w1 = m->wu[l];
        gu.n_out = c.ffn;
        gu.y = m->act;
        gu.ldy = c.ffn;
        if (fuse) gu.x = m->h;
        LAUNCH(m, K_GATEUP, st,
               mv_launch(m, gu, &wm.g, &wm.u, nullptr, &m->xmap_xn[xi], st, pdl, fuse ? m->ffn_norm[l] : nullptr));

        MatvecArgs d = {};
        d.mode = MV_RESIDUAL;
        d.K = c.ffn;
        d.n_rows = n;
        d.x = m->act;
        d.w0 = m->wd[l];
        d.n_out = H;
        d.h = m->h;
        LAUNCH(m, K_DOWN, st, mv_launch(m, d, &wm.d, nullptr, nullptr, &m->xmap_act[xi], st, pdl));
    }
    return TFL_OK;
}

// Final norm + lm_head for rows [r0, r0 + n) of m->h, n <= 64 per launch.
int run_head(tfl_model* m, int r0, int n, void* logits, long ld_rows_out, cudaStream_t st) {
    const tfl_config& c = m->cfg;
    const int H = c.hidden;
    const bool pdl = m->pdl && st != nullptr;
    for (int b = 0; b < n; b += kMaxDecodeRows) {
        const int k = std::min(kMaxDecodeRows, n - b);
        const bool fuse = k <= kMaxFusedNormRows;
        const bf16* hrows = m->h + (size_t)(r0 + b) * H;
        if (!fuse) LAUNCH(m, K_NORM, st, launch_rmsnorm(hrows, m->final_norm, c.rms_eps, k, H, m->xn, st, pdl));
        MatvecArgs a = {};
        a.mode = MV_STORE;
        a.K = H;
        a.n_rows = k;
        a.x = fuse ? hrows : m->xn;
        a.w0 = m->lm_head;
        a.n_out = c.vocab;
        a.y = (bf16*)logits + (size_t)b * ld_rows_out;
        a.ldy = ld_rows_out;
        LAUNCH(m, K_LMHEAD, st, mv_launch(m, a, &m->lm_map, nullptr, nullptr, &m->xmap_xn[xbox_index(k)], st, pdl,
                                          fuse ? m->final_norm : nullptr));
    }
    return TFL_OK;
}

int check_stream_kvs(tfl_model* m, tfl_kv* const* kvs, int n_streams, const int* rows, RowMap& rm) {
    if (!m || !kvs || !rows) return fail(TFL_E_ARG, "NULL model, kvs or rows_per_stream");
    if (n_streams < 1 || n_streams > kMaxStreams) return fail(TFL_E_ARG, "n_streams %d outside 1..16", n_streams);
    std::memset(&rm, 0, sizeof rm);
    rm.n_streams = n_streams;
    int total = 0;
    for (int s = 0; s < n_streams; ++s) {
        const tfl_kv* kv = kvs[s];
        if (!kv || kv->model != m) return fail(TFL_E_ARG, "stream %d: KV object missing or of another model", s);
        for (int t = 0; t < s; ++t)
            if (kvs[t] == kv) return fail(TFL_E_ARG, "stream %d repeats the KV object of stream %d", s, t);
        if (rows[s] < 1 || rows[s] > 16) return fail(TFL_E_ARG, "stream %d: %d rows outside 1..16", s, rows[s]);
        if (kv->length + rows[s] > kv->max_pos)
            return fail(TFL_E_CAPACITY, "stream %d: positions %d..%d reach the KV capacity %d; rejected", s,
                        kv->length, kv->length + rows[s] - 1, kv->max_pos);
        rm.row_start[s] = total;
        rm.pos0[s] = kv->length;
        rm.kv[s] = view(kv);
        total += rows[s];
    }
    rm.row_start[n_streams] = total;
    rm.n_rows = total;
    if (total > m->cfg.max_decode_rows)
        return fail(TFL_E_ARG, "%d rows in one step exceed max_decode_rows %d", total, m->cfg.max_decode_rows);
    if (total > kMaxDecodeRows) return fail(TFL_E_ARG, "%d rows exceed %d", total, kMaxDecodeRows);
    return TFL_OK;
}

// A whole decode step of at most kStepMaxRows rows as one cooperative launch.
int run_step_persistent(tfl_model* m, tfl_kv* const* kvs, const RowMap& rm, const int32_t* ids, void* logits,
                        cudaStream_t st) {
    const tfl_config& c = m->cfg;
    StepArgs a;
    std::memset(&a, 0, sizeof a);
    a.layers = c.layers;
    a.H = c.hidden;
    a.n_q = c.n_q;
    a.n_kv = c.n_kv;
    a.F = c.ffn;
    a.V = c.vocab;
    a.max_blocks = m->L.max_blocks;
    a.eps = c.rms_eps;
    a.wmaps = m->d_wmaps;
    a.norms = m->d_norms;
    a.final_norm = m->final_norm;
    a.embed = m->embed;
    a.zero_row = m->zero_row;
    a.h = m->h;
    a.q = m->q;
    a.ao = m->ao;
    a.act = m->act;
    a.pm = m->pm;
    a.pl = m->pl;
    a.po = m->po;
    a.cos_t = m->cos_t;
    a.sin_t = m->sin_t;
    a.status = m->status;
    a.sync = m->sync;
    a.ids = ids;
    a.logits = (bf16*)logits;
    a.rows = rm;
    a.attn.q = m->q;
    a.attn.out = m->ao;
    a.attn.pm = m->pm;
    a.attn.pl = m->pl;
    a.attn.po = m->po;
    a.attn.max_blocks = m->L.max_blocks;
    a.attn.n_q = c.n_q;
    a.attn.n_kv = c.n_kv;
    a.attn.rows = rm;
    for (int s = 0; s < rm.n_streams; ++s) a.kvmap[s] = kvs[s]->kvmap;
    a.ts = (m->prof && m->grid <= kStepTsCtas) ? m->ts : nullptr;
    LAUNCH(m, K_STEP, st, launch_step_persistent(a, m->grid, st));
    if (a.ts) m->ts_valid = true;
    return TFL_OK;
}

int decode_common(tfl_model* m, tfl_kv* const* kvs, int n_streams, const int* rows, const int32_t* ids,
                  const void* h_in, void* logits, void* h_out, cudaStream_t st) {
    RowMap rm;
    int e = check_stream_kvs(m, kvs, n_streams, rows, rm);
    if (e) return e;
    for (int s = 0; s < n_streams; ++s)
        if (kvs[s]->length + rows[s] > m->cfg.max_context)
            return fail(TFL_E_CAPACITY, "stream %d passes the model's max_context %d", s, m->cfg.max_context);
    if (m->persistent && ids && logits && !h_out && rm.n_rows <= kStepMaxRows) {
        e = run_step_persistent(m, kvs, rm, ids, logits, st);
        if (e) return e;
        for (int s = 0; s < n_streams; ++s) kvs[s]->length += rows[s];
        return ok();
    }
    KvMaps maps;
    for (int s = 0; s < n_streams; ++s) maps.m[s] = kvs[s]->kvmap;
    e = run_layers(m, rm, maps, ids, h_in, st);
    if (e) return e;
    if (h_out) CK(cudaMemcpyAsync(h_out, m->h, (size_t)rm.n_rows * m->cfg.hidden * 2, cudaMemcpyDeviceToDevice, st));
    if (logits) {
        e = run_head(m, 0, rm.n_rows, logits, m->cfg.vocab, st);
        if (e) return e;
    }
    for (int s = 0; s < n_streams; ++s) kvs[s]->length += rows[s];
    return ok();
}

// Launches the prompt GEMM for one projection (tiles derived from the mode).
cudaError_t gemm_launch(tfl_model* m, const MatvecArgs& e, const CUtensorMap* amap, const CUtensorMap* b0,
                        const CUtensorMap* b1, const CUtensorMap* b2, cudaStream_t st, bool pdl) {
    GemmArgs g;
    std::memset(&g, 0, sizeof g);
    g.e = e;
    g.amap = *amap;
    g.bmap[0] = *b0;
    if (b1) g.bmap[1] = *b1;
    if (b2) g.bmap[2] = *b2;
    g.m_tiles = (e.n_rows + 127) / 128;
    g.n_tiles = gemm_n_tiles(e);
    g.kblocks = e.K / 64;
    g.status = m->status;
    return launch_gemm_tc(g, m->grid, st, pdl);
}

// Causal attention of the rows of a prompt chunk (one stream, queries q,
// output out, both [rows][n_q*128]) in one launch of the prefill kernel.
int prompt_attention(tfl_model* m, const tfl_kv* kv, const RowMap& rm, int layer, const bf16* q, bf16* out,
                     cudaStream_t st, bool pdl) {
    const tfl_config& c = m->cfg;
    AttnPrefillArgs p = {};
    if (!encode_map2d(&p.qmap, q, (uint64_t)c.n_q * kHeadDim, (uint64_t)rm.n_rows, 128))
        return fail(TFL_E_ARG, "cannot describe the query rows to TMA");
    p.kvmap = kv->kvmap;
    p.status = m->status;
    p.out = out;
    p.kv = rm.kv[0];
    p.n_q = c.n_q;
    p.n_kv = c.n_kv;
    p.layer = layer;
    p.pos0 = rm.pos0[0];
    p.n_rows = rm.n_rows;
    LAUNCH(m, K_PATTN, st, launch_attn_prefill(p, st, pdl));
    return TFL_OK;
}

// The layer stack over the n rows of one prompt chunk (one stream): norms,
// tcgen05 GEMM projections with fused epilogues, attention.  Each row's result
// depends only on its own input and position, so chunk boundaries never change
// results (a prompt resumed from a kept prefix equals the same prompt fresh).
int run_prompt_layers(tfl_model* m, const tfl_kv* kv, const RowMap& rm, const int32_t* ids, const void* h_in,
                      cudaStream_t st) {
    const tfl_config& c = m->cfg;
    const int n = rm.n_rows, H = c.hidden, qd = c.n_q * kHeadDim;
    const bool pdl = m->pdl && st != nullptr;
    if (ids) {
        LAUNCH(m, K_EMBED, st,
               launch_embed_rmsnorm(ids, m->embed, c.vocab, m->attn_norm[0], c.rms_eps, n, H, m->h, m->xn, m->status,
                                    st, pdl));
    } else {
        CK(cudaMemcpyAsync(m->h, h_in, (size_t)n * H * 2, cudaMemcpyDeviceToDevice, st));
        LAUNCH(m, K_NORM, st, launch_rmsnorm(m->h, m->attn_norm[0], c.rms_eps, n, H, m->xn, st, false));
    }
    for (int l = 0; l < c.layers; ++l) {
        const tfl_model::LayerMaps& wm = m->wmaps[l];
        if (l > 0) LAUNCH(m, K_NORM, st, launch_rmsnorm(m->h, m->attn_norm[l], c.rms_eps, n, H, m->xn, st, pdl));
        MatvecArgs a = {};
        a.mode = MV_QKV_ROPE;
        a.K = H;
        a.n_rows = n;
        a.n_q = c.n_q;
        a.n_kv = c.n_kv;
        a.y = m->q;
        a.ldy = qd;
        a.cos_t = m->cos_t;
        a.sin_t = m->sin_t;
        a.layer = l;
        a.rows = rm;
        LAUNCH(m, K_GQKV, st, gemm_launch(m, a, &m->amap_xn, &wm.gq, &wm.gk, &wm.gv, st, pdl));
        int e = prompt_attention(m, kv, rm, l, m->q, m->ao, st, pdl);
        if (e) return e;
        MatvecArgs o = {};
        o.mode = MV_RESIDUAL;
        o.K = qd;
        o.n_rows = n;
        o.n_out = H;
        o.h = m->h;
        LAUNCH(m, K_GO, st, gemm_launch(m, o, &m->amap_ao, &wm.go, nullptr, nullptr, st, pdl));
        LAUNCH(m, K_NORM, st, launch_rmsnorm(m->h, m->ffn_norm[l], c.rms_eps, n, H, m->xn, st, pdl));
        MatvecArgs gu = {};
        gu.mode = MV_SWIGLU;
        gu.K = H;
        gu.n_rows = n;
        gu.n_out = c.ffn;
        gu.y = m->act;
        gu.ldy = c.ffn;
        LAUNCH(m, K_GGATEUP, st, gemm_launch(m, gu, &m->amap_xn, &wm.gg, &wm.gu, nullptr, st, pdl));
        MatvecArgs d = {};
        d.mode = MV_RESIDUAL;
        d.K = c.ffn;
        d.n_rows = n;
        d.n_out = H;
        d.h = m->h;
        LAUNCH(m, K_GDOWN, st, gemm_launch(m, d, &m->amap_act, &wm.gd, nullptr, nullptr, st, pdl));
    }
    return TFL_OK;
}

int prefill_common(tfl_model* m, tfl_kv* kv, const int32_t* ids, const void* h_in, int n_rows, void* logits,
                   int all_rows, void* h_out, cudaStream_t st) {
    if (!m || !kv || kv->model != m) return fail(TFL_E_ARG, "NULL model or KV object of another model");
    if (n_rows < 1 || n_rows > m->cfg.max_rows) return fail(TFL_E_ARG, "n_rows %d outside 1..%d", n_rows, m->cfg.max_rows);
    if (kv->length + n_rows > kv->max_pos || kv->length + n_rows > m->cfg.max_context)
        return fail(TFL_E_CAPACITY, "positions %d..%d reach the KV capacity %d; rejected", kv->length,
                    kv->length + n_rows - 1, std::min(kv->max_pos, m->cfg.max_context));
    const int H = m->cfg.hidden;
    RowMap rm;
    std::memset(&rm, 0, sizeof rm);
    rm.n_streams = 1;
    rm.n_rows = n_rows;
    rm.row_start[1] = n_rows;
    rm.pos0[0] = kv->length;
    rm.kv[0] = view(kv);
    int e = run_prompt_layers(m, kv, rm, ids, h_in, st);
    if (e) return e;
    if (h_out) CK(cudaMemcpyAsync(h_out, m->h, (size_t)n_rows * H * 2, cudaMemcpyDeviceToDevice, st));
    if (logits && all_rows) {
        e = run_head(m, 0, n_rows, logits, m->cfg.vocab, st);
        if (e) return e;
    } else if (logits) {
        e = run_head(m, n_rows - 1, 1, logits, m->cfg.vocab, st);
        if (e) return e;
    }
    kv->length += n_rows;
    return ok();
}

}  // namespace

// ---- helpers for entry points defined in other files ---------------------------------

namespace tfl {

int kv_handle_view(const tfl_kv* kv, KvView* out, int* max_pos, int* n_q, int* n_kv, int* layers) {
    if (!kv || !kv->model) return TFL_E_ARG;
    *out = view(kv);
    *max_pos = kv->max_pos;
    *n_q = kv->model->cfg.n_q;
    *n_kv = kv->model->cfg.n_kv;
    *layers = kv->model->cfg.layers;
    return TFL_OK;
}

void set_last_error(const char* msg) { g_err = msg; }

int api_fail(int code, const char* msg) { return fail(code, "%s", msg); }

int kv_prefix_geometry(const tfl_kv* kv, const tfl_model* m, bf16** pages, int* n_pages, int* length, int* max_pos) {
    if (!kv || kv->model != m) return TFL_E_ARG;
    *pages = kv->pages;
    *n_pages = kv->n_pages;
    *length = kv->length;
    *max_pos = kv->max_pos;
    return TFL_OK;
}

int kv_set_length(tfl_kv* kv, int length) {
    kv->length = length;
    return TFL_OK;
}

int model_geometry(const tfl_model* m, int* layers, int* n_kv) {
    *layers = m->cfg.layers;
    *n_kv = m->cfg.n_kv;
    return TFL_OK;
}

const tfl_config* model_config(const tfl_model* m) { return m ? &m->cfg : nullptr; }

tfl_model* kv_owner(const tfl_kv* kv) { return kv ? kv->model : nullptr; }

// Greedy ids of draft rows: a non-finite row proposes id 0 (the served model's
// check then decides) and raises the drafter's non-finite status bit.
int draft_argmax(tfl_model* m, const void* logits, int n_rows, int32_t* ids, cudaStream_t st) {
    LAUNCH(m, K_ARGMAX, st, launch_argmax((const bf16*)logits, n_rows, m->cfg.vocab, ids, m->status, st,
                                          m->pdl && st != nullptr, 0));
    return TFL_OK;
}

}  // namespace tfl

// ---- C ABI ------------------------------------------------------------------------

extern "C" {

const char* tfl_last_error(void) { return g_err.c_str(); }

const char* tfl_error_string(int code) {
    switch (code) {
        case TFL_OK: return "ok";
        case TFL_E_GEOMETRY: return "geometry not qualified";
        case TFL_E_ARCH: return "device is not sm_103";
        case TFL_E_CAPACITY: return "KV capacity reached";
        case TFL_E_ARG: return "invalid argument";
        case TFL_E_CUDA: return "CUDA error";
        case TFL_E_NONFINITE: return "non-finite logit";
        case TFL_E_WORKSPACE: return "buffer too small";
        case TFL_E_DEVICE: return "kernel gave up a bounded wait";
        default: return "unknown error";
    }
}

int tfl_qualify(const tfl_config* cfg, char* msg, size_t msg_len) {
    int e = qualify(cfg);
    if (msg && msg_len) {
        std::strncpy(msg, g_err.c_str(), msg_len - 1);
        msg[msg_len - 1] = 0;
    }
    return e;
}

size_t tfl_workspace_bytes(const tfl_config* cfg) {
    if (qualify(cfg) != TFL_OK) return 0;
    return layout(cfg).total;
}

void tfl_rope_table(double theta, int n_pos, uint16_t* cos_out, uint16_t* sin_out) {
    float inv[64];
    for (int i = 0; i < 64; ++i) {
        const float base_pow = (float)std::pow(theta, (double)(2 * i) / (double)kHeadDim);
        inv[i] = (float)(1.0 / (double)base_pow);
    }
    for (int p = 0; p < n_pos; ++p)
        for (int i = 0; i < 64; ++i) {
            const float angle = (float)((double)p * (double)inv[i]);
            cos_out[(size_t)p * 64 + i] = host_bf16(std::cos((double)angle));
            sin_out[(size_t)p * 64 + i] = host_bf16(std::sin((double)angle));
        }
}

int tfl_init(const tfl_config* cfg, const tfl_weights* w, void* workspace, size_t ws_bytes, tfl_model** out) {
    if (!out) return fail(TFL_E_ARG, "out is NULL");
    *out = nullptr;
    int e = qualify(cfg);
    if (e) return e;
    if (!w || !workspace) return fail(TFL_E_ARG, "NULL weights or workspace");
    int dev = 0;
    CK(cudaGetDevice(&dev));
    cudaDeviceProp prop;
    CK(cudaGetDeviceProperties(&prop, dev));
    if (!(prop.major == 10 && prop.minor == 3))
        return fail(TFL_E_ARCH, "this library needs an sm_103 (GB300) GPU; device %d (%s) is sm_%d%d", dev, prop.name,
                    prop.major, prop.minor);
    Layout L = layout(cfg);
    if (ws_bytes < L.total) return fail(TFL_E_WORKSPACE, "workspace %zu bytes < %zu needed", ws_bytes, L.total);
    if (!aligned16(workspace)) return fail(TFL_E_ARG, "workspace not 16-byte aligned");
    const void* globals[3] = {w->embed, w->final_norm, w->lm_head};
    for (const void* p : globals)
        if (!p || !aligned16(p)) return fail(TFL_E_ARG, "embed/final_norm/lm_head NULL or not 16-byte aligned");
    if (w->lm_head == w->embed) return fail(TFL_E_GEOMETRY, "tied heads are refused: lm_head equals embed");
    const void* const* per[9] = {w->attn_norm, w->wq, w->wk, w->wv, w->wo, w->ffn_norm, w->wg, w->wu, w->wd};
    for (int k = 0; k < 9; ++k) {
        if (!per[k]) return fail(TFL_E_ARG, "per-layer weight array %d is NULL", k);
        for (int l = 0; l < cfg->layers; ++l)
            if (!per[k][l] || !aligned16(per[k][l]))
                return fail(TFL_E_ARG, "layer %d weight %d NULL or not 16-byte aligned", l, k);
    }
    CK(init_attn_decode());
    CK(init_attn_decode_tma());

    tfl_model* m = new tfl_model();
    m->cfg = *cfg;
    m->embed = (const bf16*)w->embed;
    m->final_norm = (const bf16*)w->final_norm;
    m->lm_head = (const bf16*)w->lm_head;
    std::vector<const bf16*>* dst[9] = {&m->attn_norm, &m->wq, &m->wk, &m->wv, &m->wo,
                                        &m->ffn_norm, &m->wg, &m->wu, &m->wd};
    for (int k = 0; k < 9; ++k)
        for (int l = 0; l < cfg->layers; ++l) dst[k]->push_back((const bf16*)per[k][l]);
    m->ws = (char*)workspace;
    m->L = L;
    m->h = (bf16*)(m->ws + L.h);
    m->xn = (bf16*)(m->ws + L.xn);
    m->q = (bf16*)(m->ws + L.q);
    m->ao = (bf16*)(m->ws + L.ao);
    m->act = (bf16*)(m->ws + L.act);
    m->pm = (float*)(m->ws + L.pm);
    m->pl = (float*)(m->ws + L.pl);
    m->po = (float*)(m->ws + L.po);
    m->cos_t = (bf16*)(m->ws + L.cos_t);
    m->sin_t = (bf16*)(m->ws + L.sin_t);
    m->status = (int*)(m->ws + L.status);
    m->d_wmaps = (CUtensorMap*)(m->ws + L.wmaps);
    m->d_norms = (const bf16**)(m->ws + L.norms);
    m->sync = (unsigned*)(m->ws + L.sync);
    m->zero_row = (bf16*)(m->ws + L.zero);
    m->ts = (unsigned long long*)(m->ws + L.ts);
    m->scounts = (unsigned*)(m->ws + L.scounts);
    m->swtab = (double*)(m->ws + L.swtab);
    m->pdl = true;

    // projections: TMA descriptors of every weight matrix and activation buffer
    {
        const int H = cfg->hidden, QD = cfg->n_q * kHeadDim, KD = cfg->n_kv * kHeadDim, F = cfg->ffn;
        const size_t rows = (size_t)std::max(cfg->max_rows, cfg->max_decode_rows);
        bool okm = true;
        m->wmaps.resize(cfg->layers);
        for (int l = 0; l < cfg->layers && okm; ++l) {
            tfl_model::LayerMaps& x = m->wmaps[l];
            okm = encode_map(&x.q, m->wq[l], H, QD, 8) && encode_map(&x.k, m->wk[l], H, KD, 8) &&
                  encode_map(&x.v, m->wv[l], H, KD, 8) && encode_map(&x.o, m->wo[l], QD, H, 16) &&
                  encode_map(&x.g, m->wg[l], H, F, 8) && encode_map(&x.u, m->wu[l], H, F, 8) &&
                  encode_map(&x.d, m->wd[l], F, H, 16) &&
                  encode_map2d(&x.gq, m->wq[l], H, QD, 128) && encode_map2d(&x.gk, m->wk[l], H, KD, 128) &&
                  encode_map2d(&x.gv, m->wv[l], H, KD, 128) && encode_map2d(&x.go, m->wo[l], QD, H, 256) &&
                  encode_map2d(&x.gg, m->wg[l], H, F, 128) && encode_map2d(&x.gu, m->wu[l], H, F, 128) &&
                  encode_map2d(&x.gd, m->wd[l], F, H, 256);
        }
        okm = okm && encode_map(&m->lm_map, m->lm_head, H, cfg->vocab, 16);
        const int xrows[kXBoxes] = {1, 2, 3, 4, 5, 6, 7, 8, 16, 32, 64};
        for (int i = 0; i < kXBoxes && okm; ++i)
            okm = encode_map(&m->xmap_xn[i], m->xn, H, rows, xrows[i]) &&
                  encode_map(&m->xmap_ao[i], m->ao, QD, rows, xrows[i]) &&
                  encode_map(&m->xmap_act[i], m->act, F, rows, xrows[i]);
        okm = okm && encode_map2d(&m->amap_xn, m->xn, H, rows, 128) && encode_map2d(&m->amap_ao, m->ao, QD, rows, 128) &&
              encode_map2d(&m->amap_act, m->act, F, rows, 128);
        cudaError_t ce0 = cudaSuccess;
        if (okm) ce0 = init_matvec_tma();
        if (okm && ce0 == cudaSuccess) ce0 = init_gemm_tc();
        if (okm && ce0 == cudaSuccess) ce0 = init_attn_prefill();
        if (okm && ce0 == cudaSuccess) ce0 = init_step_persistent();
        if (okm && ce0 == cudaSuccess) {
            // device copies for the decode-step kernel: [layer][q k v o gate up down], lm_head; norms
            std::vector<CUtensorMap> dm((size_t)cfg->layers * 7 + 1);
            std::vector<const bf16*> dn((size_t)cfg->layers * 2);
            for (int l = 0; l < cfg->layers; ++l) {
                const tfl_model::LayerMaps& x = m->wmaps[l];
                const CUtensorMap seven[7] = {x.q, x.k, x.v, x.o, x.g, x.u, x.d};
                for (int j = 0; j < 7; ++j) dm[(size_t)l * 7 + j] = seven[j];
                dn[(size_t)l * 2] = m->attn_norm[l];
                dn[(size_t)l * 2 + 1] = m->ffn_norm[l];
            }
            dm.back() = m->lm_map;
            ce0 = cudaMemcpy(m->d_wmaps, dm.data(), dm.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice);
            if (ce0 == cudaSuccess)
                ce0 = cudaMemcpy(m->d_norms, dn.data(), dn.size() * sizeof(void*), cudaMemcpyHostToDevice);
            if (ce0 == cudaSuccess) ce0 = cudaMemset(m->zero_row, 0, (size_t)cfg->hidden * 2);
            if (ce0 == cudaSuccess) ce0 = cudaMemset(m->sync, 0, 256);
        }
        if (!okm || ce0 != cudaSuccess) {
            delete m;
            return fail(TFL_E_CUDA, "building TMA descriptors failed%s%s", ce0 ? ": " : "",
                        ce0 ? cudaGetErrorString(ce0) : "");
        }
        m->grid = prop.multiProcessorCount;
    }

    std::vector<uint16_t> c((size_t)cfg->max_context * 64), s((size_t)cfg->max_context * 64);
    tfl_rope_table(cfg->rope_theta, cfg->max_context, c.data(), s.data());
    cudaError_t ce = cudaMemcpy(m->cos_t, c.data(), c.size() * 2, cudaMemcpyHostToDevice);
    if (ce == cudaSuccess) ce = cudaMemcpy(m->sin_t, s.data(), s.size() * 2, cudaMemcpyHostToDevice);
    if (ce == cudaSuccess) ce = cudaMemset(m->status, 0, 256);
    // sampling counts start at zero; every tfl_sample call leaves them zero again
    if (ce == cudaSuccess) ce = cudaMemset(m->scounts, 0, (size_t)cfg->max_decode_rows * 65536 * 4);
    if (ce != cudaSuccess) {
        delete m;
        return fail(TFL_E_CUDA, "uploading the RoPE table failed: %s", cudaGetErrorString(ce));
    }
    *out = m;
    return ok();
}

void tfl_free(tfl_model* m) { delete m; }

int tfl_step_phases(tfl_model* m, double* out, int n) {
    if (!m || !out || n < 9) return fail(TFL_E_ARG, "NULL model or output, or n < 9");
    if (!m->ts_valid) return fail(TFL_E_ARG, "no profiled persistent decode step since the last tfl_step_phases");
    const int L = m->cfg.layers, stride = step_ts_stride(L), G = m->grid;
    std::vector<unsigned long long> t((size_t)G * stride);
    CK(cudaDeviceSynchronize());
    CK(cudaMemcpy(t.data(), m->ts, t.size() * 8, cudaMemcpyDeviceToHost));
    m->ts_valid = false;
    auto at = [&](int c, int i) { return (double)t[(size_t)c * stride + i]; };
    auto cmax = [&](int i) { double v = at(0, i); for (int c = 1; c < G; ++c) v = std::max(v, at(c, i)); return v; };
    auto cmin = [&](int i) { double v = at(0, i); for (int c = 1; c < G; ++c) v = std::min(v, at(c, i)); return v; };
    for (int k = 0; k < 9; ++k) out[k] = 0.0;
    double prev = cmax(0), bar_sum = 0.0;
    for (int e = 1; e <= 6 * L; ++e) {
        const double pass = cmax(2 * e + 1);
        out[(e - 1) % 6] += (pass - prev) / 1e3 / L;
        bar_sum += (cmin(2 * e + 1) - cmax(2 * e)) / 1e3;
        prev = pass;
    }
    out[6] = bar_sum / (6.0 * L);
    out[7] = (cmax(1) - prev) / 1e3;
    out[8] = (cmax(1) - cmin(0)) / 1e3;
    return ok();
}

int tfl_set_persistent(tfl_model* m, int enable) {
    if (!m) return fail(TFL_E_ARG, "NULL model");
    m->persistent = enable != 0;
    return ok();
}

size_t tfl_kv_bytes(const tfl_config* cfg, int max_positions) {
    if (!cfg || max_positions < 1 || cfg->n_kv < 1 || cfg->layers < 1) return 0;
    const int n_pages = (max_positions + kPage - 1) / kPage;
    return kv_table_bytes(n_pages) +
           (size_t)cfg->layers * 2 * n_pages * kPage * (size_t)cfg->n_kv * kHeadDim * 2;
}

int tfl_kv_alloc(tfl_model* m, int max_positions, void* dev_buf, size_t bytes, tfl_kv** out) {
    if (!out) return fail(TFL_E_ARG, "out is NULL");
    *out = nullptr;
    if (!m || !dev_buf) return fail(TFL_E_ARG, "NULL model or buffer");
    if (max_positions < 1 || max_positions > m->cfg.max_context)
        return fail(TFL_E_ARG, "max_positions %d outside 1..max_context %d", max_positions, m->cfg.max_context);
    if (!aligned16(dev_buf)) return fail(TFL_E_ARG, "KV buffer not 16-byte aligned");
    const size_t need = tfl_kv_bytes(&m->cfg, max_positions);
    if (bytes < need) return fail(TFL_E_WORKSPACE, "KV buffer %zu bytes < %zu needed", bytes, need);
    tfl_kv* kv = new tfl_kv();
    kv->model = m;
    kv->buf = (char*)dev_buf;
    kv->max_pos = max_positions;
    kv->n_pages = (max_positions + kPage - 1) / kPage;
    kv->length = 0;
    kv->table = (int*)dev_buf;
    kv->pages = (bf16*)((char*)dev_buf + kv_table_bytes(kv->n_pages));
    if (!encode_kv_map(&kv->kvmap, kv->pages, m->cfg.n_kv,
                       (uint64_t)m->cfg.layers * 2 * (uint64_t)kv->n_pages * kPage)) {
        delete kv;
        return fail(TFL_E_CUDA, "building the KV tensor map failed");
    }
    std::vector<int> ident(kv->n_pages);
    for (int i = 0; i < kv->n_pages; ++i) ident[i] = i;
    cudaError_t ce = cudaMemcpy(kv->table, ident.data(), ident.size() * 4, cudaMemcpyHostToDevice);
    if (ce != cudaSuccess) {
        delete kv;
        return fail(TFL_E_CUDA, "writing the page table failed: %s", cudaGetErrorString(ce));
    }
    *out = kv;
    return ok();
}

void tfl_kv_free(tfl_kv* kv) { delete kv; }

int tfl_kv_reset(tfl_kv* kv, int keep) {
    if (!kv) return fail(TFL_E_ARG, "NULL KV object");
    if (keep < 0 || keep > kv->max_pos) return fail(TFL_E_ARG, "keep %d outside 0..%d", keep, kv->max_pos);
    kv->length = keep;
    return ok();
}

int tfl_kv_length(const tfl_kv* kv) { return kv ? kv->length : -1; }
int tfl_kv_capacity(const tfl_kv* kv) { return kv ? kv->max_pos : -1; }

static int kv_copy(tfl_model* m, const tfl_kv* kv, int layer, int pos0, int n, void* k, void* v, bool to_cache,
                   void* stream) {
    if (!m || !kv || kv->model != m || !k || !v) return fail(TFL_E_ARG, "NULL argument or KV of another model");
    if (layer < 0 || layer >= m->cfg.layers) return fail(TFL_E_ARG, "layer %d outside 0..%d", layer, m->cfg.layers - 1);
    if (n < 0 || pos0 < 0 || pos0 + n > kv->max_pos)
        return fail(TFL_E_ARG, "positions %d..%d outside the capacity %d", pos0, pos0 + n - 1, kv->max_pos);
    if (!aligned16(k) || !aligned16(v)) return fail(TFL_E_ARG, "k/v not 16-byte aligned");
    CK(launch_kv_copy(kv->pages, kv->table, kv->n_pages, m->cfg.n_kv, layer, pos0, n, (bf16*)k, (bf16*)v, to_cache,
                      (cudaStream_t)stream));
    return ok();
}

int tfl_kv_write(tfl_model* m, tfl_kv* kv, int layer, int pos0, int n, const void* k, const void* v, void* stream) {
    return kv_copy(m, kv, layer, pos0, n, (void*)k, (void*)v, true, stream);
}

int tfl_kv_read(tfl_model* m, const tfl_kv* kv, int layer, int pos0, int n, void* k, void* v, void* stream) {
    return kv_copy(m, kv, layer, pos0, n, k, v, false, stream);
}

int tfl_decode_step(tfl_model* m, tfl_kv* const* kvs, int n_streams, const int32_t* ids, const int* rows,
                    void* logits, void* stream) {
    if (!ids || !logits) return fail(TFL_E_ARG, "NULL ids or logits");
    return decode_common(m, kvs, n_streams, rows, ids, nullptr, logits, nullptr, (cudaStream_t)stream);
}

int tfl_decode_hidden(tfl_model* m, tfl_kv* const* kvs, int n_streams, const int* rows, const void* h_in,
                      void* h_out, void* stream) {
    if (!h_in || !h_out) return fail(TFL_E_ARG, "NULL h_in or h_out");
    return decode_common(m, kvs, n_streams, rows, nullptr, h_in, nullptr, h_out, (cudaStream_t)stream);
}

int tfl_prefill_chunk(tfl_model* m, tfl_kv* kv, const int32_t* ids, int n_rows, void* logits, int all_rows,
                      void* stream) {
    if (!ids) return fail(TFL_E_ARG, "NULL ids");
    return prefill_common(m, kv, ids, nullptr, n_rows, logits, all_rows, nullptr, (cudaStream_t)stream);
}

int tfl_prefill_hidden(tfl_model* m, tfl_kv* kv, const void* h_in, int n_rows, void* h_out, void* stream) {
    if (!h_in || !h_out) return fail(TFL_E_ARG, "NULL h_in or h_out");
    return prefill_common(m, kv, nullptr, h_in, n_rows, nullptr, 0, h_out, (cudaStream_t)stream);
}

int tfl_head(tfl_model* m, const void* h, int rows, void* logits, void* stream) {
    if (!m || !h || !logits) return fail(TFL_E_ARG, "NULL argument");
    if (rows < 1 || rows > std::max(m->cfg.max_rows, m->cfg.max_decode_rows))
        return fail(TFL_E_ARG, "rows %d outside 1..%d", rows, std::max(m->cfg.max_rows, m->cfg.max_decode_rows));
    cudaStream_t st = (cudaStream_t)stream;
    CK(cudaMemcpyAsync(m->h, h, (size_t)rows * m->cfg.hidden * 2, cudaMemcpyDeviceToDevice, st));
    int e = run_head(m, 0, rows, logits, m->cfg.vocab, st);
    return e ? e : ok();
}

int tfl_sample(tfl_model* m, const void* logits, int n_rows, float temperature, int top_k, float top_p,
               const float* u, int32_t* ids, void* stream) {
    if (!m || !logits || !u || !ids) return fail(TFL_E_ARG, "NULL model, logits, u or ids");
    if (n_rows < 1 || n_rows > m->cfg.max_decode_rows)
        return fail(TFL_E_ARG, "n_rows %d outside 1..max_decode_rows %d", n_rows, m->cfg.max_decode_rows);
    if (!(temperature > 0.f) || !std::isfinite(temperature))
        return fail(TFL_E_ARG, "temperature %g must be finite and > 0 (use tfl_argmax for greedy)", (double)temperature);
    if (top_k < 0) return fail(TFL_E_ARG, "top_k %d < 0", top_k);
    if (!(top_p > 0.f) || std::isnan(top_p)) return fail(TFL_E_ARG, "top_p %g must be > 0", (double)top_p);
    if (((uintptr_t)logits & 1u) || ((uintptr_t)u & 3u) || ((uintptr_t)ids & 3u))
        return fail(TFL_E_ARG, "misaligned logits, u or ids");
    cudaStream_t st = (cudaStream_t)stream;
    LAUNCH(m, K_SAMPLE, st,
           launch_sample((const bf16*)logits, n_rows, m->cfg.vocab, temperature, top_k, top_p, u, ids, m->status,
                         m->scounts, m->swtab, st, m->pdl && st != nullptr));
    return ok();
}

int tfl_argmax(tfl_model* m, const void* logits, int n_rows, int32_t* ids, void* stream) {
    if (!m || !logits || !ids) return fail(TFL_E_ARG, "NULL argument");
    if (n_rows < 1) return fail(TFL_E_ARG, "n_rows %d < 1", n_rows);
    cudaStream_t st = (cudaStream_t)stream;
    LAUNCH(m, K_ARGMAX, st, launch_argmax((const bf16*)logits, n_rows, m->cfg.vocab, ids, m->status, st, m->pdl && st != nullptr));
    return ok();
}

int tfl_layer_op(tfl_model* m, int op, int layer, tfl_kv* kv, int pos0, int rows, const void* in, void* out,
                 void* stream) {
    if (!m || !in || !out) return fail(TFL_E_ARG, "NULL model, in or out");
    const tfl_config& c = m->cfg;
    const bool prompt = (op & TFL_OP_PROMPT) != 0;
    op &= ~TFL_OP_PROMPT;
    if (op < TFL_OP_ATTN_NORM || op > TFL_OP_NORM_LM_HEAD) return fail(TFL_E_ARG, "unknown op %d", op);
    const bool no_layer = op == TFL_OP_FINAL_NORM || op == TFL_OP_LM_HEAD || op == TFL_OP_NORM_LM_HEAD;
    if (!no_layer && (layer < 0 || layer >= c.layers))
        return fail(TFL_E_ARG, "layer %d outside 0..%d", layer, c.layers - 1);
    if (prompt && (op == TFL_OP_LM_HEAD || op == TFL_OP_NORM_LM_HEAD))
        return fail(TFL_E_ARG, "the prompt path computes logits with the decode head; run op %d without TFL_OP_PROMPT", op);
    const int max_r = prompt ? c.max_rows : c.max_decode_rows;
    if (rows < 1 || rows > max_r) return fail(TFL_E_ARG, "rows %d outside 1..%d", rows, max_r);
    if (!aligned16(in) || !aligned16(out)) return fail(TFL_E_ARG, "in/out not 16-byte aligned");
    const bool uses_kv = op == TFL_OP_QKV_ROPE || op == TFL_OP_ATTENTION || op == TFL_OP_NORM_QKV_ROPE;
    RowMap rm;
    std::memset(&rm, 0, sizeof rm);
    if (uses_kv) {
        if (!kv || kv->model != m) return fail(TFL_E_ARG, "op %d needs a KV object of this model", op);
        if (pos0 < 0 || pos0 + rows > kv->max_pos)
            return fail(TFL_E_CAPACITY, "positions %d..%d outside the capacity %d", pos0, pos0 + rows - 1, kv->max_pos);
        rm.n_streams = 1;
        rm.n_rows = rows;
        rm.row_start[1] = rows;
        rm.pos0[0] = pos0;
        rm.kv[0] = view(kv);
    }
    cudaStream_t st = (cudaStream_t)stream;
    const int H = c.hidden, qd = c.n_q * kHeadDim;
    MatvecArgs a = {};
    a.n_rows = rows;
    a.x = (const bf16*)in;
    // the caller's activation rows as a TMA source (rows beyond `rows` read as zeros)
    CUtensorMap xm;
    auto xmap = [&](int K) {
        return encode_map(&xm, in, (uint64_t)K, (uint64_t)rows, (uint32_t)matvec_tma_x_rows(rows));
    };
    // ... or as the A operand of the prompt GEMM (128-row boxes)
    auto amap = [&](int K) { return encode_map2d(&xm, in, (uint64_t)K, (uint64_t)rows, 128); };
    // fused norm + projection: in is the residual stream; more than 8 rows run the
    // norm kernel into the workspace first, then the projection reads it by TMA
    const bool fused_op = op == TFL_OP_NORM_QKV_ROPE || op == TFL_OP_NORM_GATE_UP || op == TFL_OP_NORM_LM_HEAD;
    const bf16* norm_w = nullptr;
    if (fused_op) {
        const bf16* w = op == TFL_OP_NORM_QKV_ROPE ? m->attn_norm[layer]
                      : op == TFL_OP_NORM_GATE_UP ? m->ffn_norm[layer] : m->final_norm;
        if (rows <= kMaxFusedNormRows && !prompt) {
            norm_w = w;
        } else {
            LAUNCH(m, K_NORM, st, launch_rmsnorm((const bf16*)in, w, c.rms_eps, rows, H, m->xn, st, false));
            a.x = m->xn;
            in = m->xn;
        }
        op = op == TFL_OP_NORM_QKV_ROPE ? TFL_OP_QKV_ROPE : op == TFL_OP_NORM_GATE_UP ? TFL_OP_GATE_UP : TFL_OP_LM_HEAD;
    }
    switch (op) {
        case TFL_OP_ATTN_NORM:
        case TFL_OP_FFN_NORM:
        case TFL_OP_FINAL_NORM: {
            const bf16* w = op == TFL_OP_ATTN_NORM ? m->attn_norm[layer]
                          : op == TFL_OP_FFN_NORM ? m->ffn_norm[layer] : m->final_norm;
            LAUNCH(m, K_NORM, st, launch_rmsnorm((const bf16*)in, w, c.rms_eps, rows, H, (bf16*)out, st, false));
            break;
        }
        case TFL_OP_QKV_ROPE:
            a.mode = MV_QKV_ROPE;
            a.K = H;
            a.w0 = m->wq[layer];
            a.w1 = m->wk[layer];
            a.w2 = m->wv[layer];
            a.n_q = c.n_q;
            a.n_kv = c.n_kv;
            a.y = (bf16*)out;
            a.ldy = qd;
            a.cos_t = m->cos_t;
            a.sin_t = m->sin_t;
            a.layer = layer;
            a.rows = rm;
            if (prompt) {
                if (!amap(H)) return fail(TFL_E_ARG, "cannot describe the input rows to TMA");
                LAUNCH(m, K_GQKV, st,
                       gemm_launch(m, a, &xm, &m->wmaps[layer].gq, &m->wmaps[layer].gk, &m->wmaps[layer].gv, st,
                                   false));
                break;
            }
            if (!xmap(H)) return fail(TFL_E_ARG, "cannot describe the input rows to TMA");
            LAUNCH(m, K_QKV, st,
                   mv_launch(m, a, &m->wmaps[layer].q, &m->wmaps[layer].k, &m->wmaps[layer].v, &xm, st, false,
                             norm_w));
            break;
        case TFL_OP_ATTENTION: {
            AttnDecodeArgs at = {};
            at.q = (const bf16*)in;
            at.out = (bf16*)out;
            at.pm = m->pm;
            at.pl = m->pl;
            at.po = m->po;
            at.max_blocks = m->L.max_blocks;
            at.n_q = c.n_q;
            at.n_kv = c.n_kv;
            at.layer = layer;
            at.rows = rm;
            if (prompt) {
                const int e = prompt_attention(m, kv, rm, layer, (const bf16*)in, (bf16*)out, st, false);
                if (e) return e;
                break;
            }
            KvMaps maps;
            maps.m[0] = kv->kvmap;
            LAUNCH(m, K_ATTN, st, launch_attn_decode(m, at, maps, st, false));
            LAUNCH(m, K_MERGE, st, launch_attn_merge(at, st, false));
            break;
        }
        case TFL_OP_O_RESIDUAL:
        case TFL_OP_DOWN_RESIDUAL:
            a.mode = MV_RESIDUAL;
            a.K = op == TFL_OP_O_RESIDUAL ? qd : c.ffn;
            a.w0 = op == TFL_OP_O_RESIDUAL ? m->wo[layer] : m->wd[layer];
            a.n_out = H;
            a.h = (bf16*)out;
            if (prompt) {
                if (!amap(a.K)) return fail(TFL_E_ARG, "cannot describe the input rows to TMA");
                LAUNCH(m, op == TFL_OP_O_RESIDUAL ? K_GO : K_GDOWN, st,
                       gemm_launch(m, a, &xm, op == TFL_OP_O_RESIDUAL ? &m->wmaps[layer].go : &m->wmaps[layer].gd,
                                   nullptr, nullptr, st, false));
                break;
            }
            if (!xmap(a.K)) return fail(TFL_E_ARG, "cannot describe the input rows to TMA");
            LAUNCH(m, op == TFL_OP_O_RESIDUAL ? K_O : K_DOWN, st,
                   mv_launch(m, a, op == TFL_OP_O_RESIDUAL ? &m->wmaps[layer].o : &m->wmaps[layer].d, nullptr,
                             nullptr, &xm, st, false));
            break;
        case TFL_OP_GATE_UP:
            a.mode = MV_SWIGLU;
            a.K = H;
            a.w0 = m->wg[layer];
            a.w1 = m->wu[layer];
            a.n_out = c.ffn;
            a.y = (bf16*)out;
            a.ldy = c.ffn;
            if (prompt) {
                if (!amap(H)) return fail(TFL_E_ARG, "cannot describe the input rows to TMA");
                LAUNCH(m, K_GGATEUP, st,
                       gemm_launch(m, a, &xm, &m->wmaps[layer].gg, &m->wmaps[layer].gu, nullptr, st, false));
                break;
            }
            if (!xmap(H)) return fail(TFL_E_ARG, "cannot describe the input rows to TMA");
            LAUNCH(m, K_GATEUP, st,
                   mv_launch(m, a, &m->wmaps[layer].g, &m->wmaps[layer].u, nullptr, &xm, st, false, norm_w));
            break;
        case TFL_OP_LM_HEAD:
            a.mode = MV_STORE;
            a.K = H;
            a.w0 = m->lm_head;
            a.n_out = c.vocab;
            a.y = (bf16*)out;
            a.ldy = c.vocab;
            if (!xmap(H)) return fail(TFL_E_ARG, "cannot describe the input rows to TMA");
            LAUNCH(m, K_LMHEAD, st, mv_launch(m, a, &m->lm_map, nullptr, nullptr, &xm, st, false, norm_w));
            break;
    }
    return ok();
}

int tfl_profile(tfl_model* m, int enable) {
    if (!m) return fail(TFL_E_ARG, "NULL model");
    m->prof = enable != 0;
    return ok();
}

int tfl_profile_read(tfl_model* m, int n_kinds, double* ms, long* launches) {
    if (!m || n_kinds < 0 || (n_kinds > 0 && (!ms || !launches))) return fail(TFL_E_ARG, "bad arguments");
    for (int k = 0; k < n_kinds; ++k) {
        ms[k] = 0.0;
        launches[k] = 0;
    }
    CK(cudaDeviceSynchronize());
    for (Mark& k : m->marks) {
        float t = 0.f;
        CK(cudaEventElapsedTime(&t, k.a, k.b));
        if (k.kind < n_kinds) {
            ms[k.kind] += t;
            launches[k.kind] += 1;
        }
        m->spare.push_back(k.a);
        m->spare.push_back(k.b);
    }
    m->marks.clear();
    return ok();
}

const char* tfl_profile_kind(int kind) { return (kind >= 0 && kind < K_COUNT) ? kKindName[kind] : nullptr; }

int tfl_wait_probe(tfl_model* m, int which, int spin_limit, void* stream) {
    if (!m) return fail(TFL_E_ARG, "NULL model");
    if (which != 0 && which != 1) return fail(TFL_E_ARG, "which %d: 0 (grid barrier) or 1 (mbarrier)", which);
    if (spin_limit < 1 || spin_limit > (1 << 20))
        return fail(TFL_E_ARG, "spin_limit %d outside 1..%d", spin_limit, 1 << 20);
    CK(launch_wait_probe(m->sync, m->status, which, (uint32_t)spin_limit, m->grid, (cudaStream_t)stream));
    return ok();
}

int tfl_status(tfl_model* m, void* stream) {
    if (!m) return fail(TFL_E_ARG, "NULL model");
    cudaStream_t st = (cudaStream_t)stream;
    CK(cudaStreamSynchronize(st));
    int s = 0;
    CK(cudaMemcpy(&s, m->status, 4, cudaMemcpyDeviceToHost));
    CK(cudaMemset(m->status, 0, 4));
    if (s & kStatusDevice) return fail(TFL_E_DEVICE, "a kernel gave up a bounded wait");
    if (s & kStatusNonFinite) return fail(TFL_E_NONFINITE, "an argmax row held NaN or +-Inf");
    if (s & kStatusBadToken) return fail(TFL_E_ARG, "a token id was outside [0, vocab)");
    return ok();
}

}  // extern "C"
