// Internal declarations shared by the sm_103a kernels and the host orchestrator.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace tfl {

typedef __nv_bfloat16 bf16;

constexpr int kHeadDim = 128;      // D: the only head size the library serves
constexpr int kPage = 128;          // KV positions per page
constexpr int kAttnUnit = 4 * kPage;  // keys per decode-attention partial (512)
constexpr int kMaxStreams = 16;    // streams in one decode step
constexpr int kMaxDecodeRows = 64; // rows in one decode step, over all streams
constexpr int kMaxChunkRows = 2048;

// Device status word bits (read and cleared by tfl_status).
constexpr int kStatusNonFinite = 1;  // an argmax row held NaN / +-Inf
constexpr int kStatusBadToken = 2;   // a token id outside [0, vocab)
constexpr int kStatusDevice = 4;     // a bounded wait gave up

// One stream's paged cache: K(layer,pos) / V(layer,pos) rows of n_kv*D bf16.
struct KvView {
    bf16* pages;       // first page
    const int* table;  // logical page -> physical page
    int n_pages;
    int pad_;
};

// Rows of one call, grouped by stream: rows [row_start[s], row_start[s+1])
// belong to stream s and sit at positions pos0[s], pos0[s]+1, ...
struct RowMap {
    int n_streams;
    int n_rows;
    int row_start[kMaxStreams + 1];
    int pos0[kMaxStreams];
    KvView kv[kMaxStreams];
};

__device__ __forceinline__ int row_stream(const RowMap& m, int r) {
    int s = 0;
    while (s + 1 < m.n_streams && r >= m.row_start[s + 1]) ++s;
    return s;
}

__device__ __forceinline__ bf16* kv_row(const KvView& v, int layer, int kind, int pos, int n_kv) {
    int page = __ldg(v.table + pos / kPage);
    size_t idx = (((size_t)(layer * 2 + kind) * v.n_pages + page) * kPage + pos % kPage) * (size_t)n_kv * kHeadDim;
    return v.pages + idx;
}

__device__ __forceinline__ float bf(bf16 x) { return __bfloat162float(x); }
__device__ __forceinline__ bf16 rn(float x) { return __float2bfloat16_rn(x); }
__device__ __forceinline__ float rbf(float x) { return __bfloat162float(__float2bfloat16_rn(x)); }

// Programmatic dependent launch: wait for the grids this one depends on (no-op
// when launched without the attribute), and allow dependents to start.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- kernel launchers (each returns the cudaError_t of its launch) ----------

// Epilogues of the decode matvec (fused into the projection).
enum MatvecMode { MV_STORE = 0, MV_RESIDUAL = 1, MV_SWIGLU = 2, MV_QKV_ROPE = 3 };

struct MatvecArgs {
    int mode;
    int K;                 // reduction length (multiple of 256)
    int n_rows;            // activation rows, 1..64
    const bf16* x;         // [n_rows][K]
    // weights (the TMA kernel reads them through its tensor maps): STORE/RESIDUAL
    // w0 ([N][K]); SWIGLU w0 = gate, w1 = up ([F][K]); QKV_ROPE w0 = Wq, w1 = Wk, w2 = Wv.
    const bf16* w0;
    const bf16* w1;
    const bf16* w2;
    int n_out;             // STORE/RESIDUAL: N; SWIGLU: F; QKV: unused
    int n_q, n_kv;         // QKV heads
    bf16* y;               // STORE: [n_rows][ldy]; SWIGLU: [n_rows][F]; QKV: q out [n_rows][n_q*D]
    long ldy;
    bf16* h;               // RESIDUAL: [n_rows][N] updated in place
    const bf16* cos_t;     // QKV: [positions][64]
    const bf16* sin_t;
    int layer;             // QKV: cache layer
    RowMap rows;           // QKV: positions and caches of the rows
};

// The TMA-fed variant: weights through 3-D tensor maps over [N][K] viewed as
// (64 columns, rows, K/64 k-blocks) with 128-byte swizzle and boxes of
// (64, 16 or 8 rows, 8 k-blocks); activation rows likewise with boxes of
// (64, x_rows_box, 8).
struct MatvecTmaArgs {
    MatvecArgs e;           // mode, K, n_rows, epilogue outputs, positions
    CUtensorMap wmap[3];    // STORE/RESIDUAL [0] (16-row boxes); SWIGLU gate, up; QKV q, k, v (8-row boxes)
    CUtensorMap xmap;       // activation rows, box rows = x_rows_box
    int x_rows_box;         // n_rows for n_rows <= 8, else 8 * NT
    int tiles;              // tiles of 16 weight rows
    int kstages;            // ceil(K / 512)
    int* status;
    // fused RMSNorm (up to 8 rows, K = hidden): e.x is the residual stream and
    // the kernel normalises it with norm_w; xmap is unused
    const bf16* norm_w;
    float eps;
    int depth;              // ring stages of the fused-norm variant (matvec_norm_depth)
};
int matvec_tma_nt(int n_rows);
int matvec_tma_x_rows(int n_rows);
int matvec_tma_tiles(const MatvecArgs& e);
cudaError_t init_matvec_tma();
int matvec_norm_depth(int n_rows, int K);
cudaError_t launch_matvec_tma(const MatvecTmaArgs& a, int grid, cudaStream_t st, bool pdl);

// Prompt-chunk GEMM on tcgen05: activations [rows][K] through a 2-D map with
// boxes of (64, 128 rows); weights 2-D with boxes of (64, 256) for STORE /
// RESIDUAL, (64, 128) = one head for QKV_ROPE, (64, 64) for the gate and up
// halves of SWIGLU.  e.n_rows is the chunk's row count; rows sit at positions
// e.rows.pos0[0] + r of stream 0.
struct GemmArgs {
    MatvecArgs e;
    CUtensorMap amap;
    CUtensorMap bmap[3];
    int m_tiles, n_tiles, kblocks;
    int* status;
};
cudaError_t init_gemm_tc();
int gemm_tile_n(int mode);
int gemm_n_tiles(const MatvecArgs& e);  // output tiles of a projection, -1 if the shape does not tile
cudaError_t launch_gemm_tc(const GemmArgs& a, int grid, cudaStream_t st, bool pdl);

cudaError_t launch_embed_rmsnorm(const int32_t* ids, const bf16* embed, int vocab, const bf16* w, float eps,
                                 int n_rows, int H, bf16* h, bf16* xn, int* status, cudaStream_t st, bool pdl);
cudaError_t launch_rmsnorm(const bf16* x, const bf16* w, float eps, int n_rows, int H, bf16* out,
                           cudaStream_t st, bool pdl);

struct AttnDecodeArgs {
    const bf16* q;        // [n_rows][n_q*D] rotated
    bf16* out;            // [n_rows][n_q*D]
    float* pm;            // [n_rows][n_q][max_blocks]
    float* pl;
    float* po;            // [n_rows][n_q][max_blocks][D]
    int max_blocks;
    int n_q, n_kv, layer;
    RowMap rows;
};
cudaError_t init_attn_decode();
cudaError_t launch_attn_block(const AttnDecodeArgs& a, cudaStream_t st, bool pdl);
cudaError_t launch_attn_merge(const AttnDecodeArgs& a, cudaStream_t st, bool pdl);

// Causal attention of the rows of one prompt chunk (one stream): row r at
// position pos0 + r attends keys 0 .. pos0 + r of kv (layer).
struct AttnPrefillArgs {
    CUtensorMap qmap;     // q [n_rows][n_q*D] rotated: 2-D, boxes of 64 columns x 128 rows, 128-byte swizzle
    CUtensorMap kvmap;    // the cache's pages (the tfl_kv's 3-D map: 64 dims x 1 head x 128 positions)
    bf16* out;            // [n_rows][n_q*D]
    KvView kv;
    int n_q, n_kv, layer;
    int pos0, n_rows;
    int* status;
};
cudaError_t init_attn_prefill();
cudaError_t launch_attn_prefill(const AttnPrefillArgs& a, cudaStream_t st, bool pdl);

// One whole decode step (embedding, every layer, final norm and lm_head) of at
// most kStepMaxRows rows as one cooperative launch (step_persistent.cu).
constexpr int kStepMaxRows = 2;
struct StepArgs {
    int layers, H, n_q, n_kv, F, V, max_blocks;
    float eps;
    const CUtensorMap* wmaps;   // device: [layers][7] (q, k, v, o, gate, up, down), then lm_head
    const bf16* const* norms;   // device: [layers][2] (attention norm, FFN norm)
    const bf16* final_norm;
    const bf16* embed;
    const bf16* zero_row;       // H zeros (the row of an out-of-range id)
    bf16 *h, *q, *ao, *act;
    float *pm, *pl, *po;
    const bf16 *cos_t, *sin_t;
    int* status;
    unsigned* sync;             // [0] grid barrier counter (zero at launch), [1] abort flag
    const int32_t* ids;         // device, n_rows
    bf16* logits;               // device [n_rows][V]
    RowMap rows;
    AttnDecodeArgs attn;        // the attention's view of q, ao, the partials and rows (layer unused)
    unsigned long long* ts;     // optional (NULL: off): per CTA, kStepTsStride global-timer stamps
    CUtensorMap kvmap[kStepMaxRows];  // per stream: 3-D map over the cache pages (128 dims, n_kv, rows)
};
// Phase stamps of the decode-step kernel, per CTA: [0] start, [1] end, then for
// grid barrier e = 1, 2, ...: [2e] arrival, [2e+1] pass.
constexpr int kStepTsCtas = 160;
__host__ __device__ inline int step_ts_stride(int layers) { return 2 + 2 * 6 * layers; }
int step_smem_bytes(int rows);
cudaError_t init_step_persistent();
cudaError_t launch_step_persistent(const StepArgs& a, int grid, cudaStream_t st);
// The step kernel's bounded waits alone on events that never happen (which = 0:
// grid barrier over `grid` CTAs; 1: mbarrier), giving up after `limit` polls.
cudaError_t launch_wait_probe(unsigned* sync, int* status, int which, uint32_t limit, int grid, cudaStream_t st);

// Seeded sampling (sample.cu); counts / wtab: per row 65,536 unsigned / double of scratch.
cudaError_t launch_sample(const bf16* logits, int n_rows, int V, float temperature, int top_k, float top_p,
                          const float* u, int32_t* ids, int* status, unsigned* counts, double* wtab, cudaStream_t st,
                          bool pdl);

// Greedy id per row (ties to the lower id); a row holding NaN / +-Inf gets
// bad_id (-1 for callers, 0 for a draft, which the served model then checks)
// and raises kStatusNonFinite.
cudaError_t launch_argmax(const bf16* logits, int n_rows, int V, int32_t* ids, int* status, cudaStream_t st,
                          bool pdl, int bad_id = -1);

cudaError_t launch_kv_copy(bf16* cache_pages, const int* table, int n_pages, int n_kv, int layer, int pos0, int n,
                           bf16* k, bf16* v, bool to_cache, cudaStream_t st);

}  // namespace tfl
