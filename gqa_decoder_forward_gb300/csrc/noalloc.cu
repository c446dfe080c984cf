// Decode attention without any caller-provided scratch: the per-block softmax
// partials live in a fixed array in the library's own device memory.
//
// Who needs this: callers that cannot allocate device memory at the point they
// run attention, for example a serving runtime whose memory manager reserves
// the whole GPU up front and hands out no extra buffers, or code that must not
// call cudaMalloc/cudaFree because those calls can synchronise the device (and
// are not allowed while a stream is being captured).  They pass only the
// queries, the KV cache and the output; this entry point allocates nothing.
//
// Limits and sharing: the array holds kScratchBytes (16 MiB) on every GPU that
// loads the library, for the life of the process.  Every call uses the same
// array, so calls that overlap on the GPU (for example on two streams at once)
// race and must be serialised by the caller.  Nothing in it needs clearing: a
// call reads only partials it has written itself.
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "../../include/tfl.h"

namespace tfl {
int kv_handle_view(const tfl_kv* kv, KvView* out, int* max_pos, int* n_q, int* n_kv, int* layers);
void set_last_error(const char* msg);
}  // namespace tfl

namespace {

constexpr size_t kScratchBytes = 16u << 20;
constexpr int kUnitFloats = tfl::kHeadDim + 2;  // o[128], m, l per (row, head, block)
constexpr size_t kMaxUnits = kScratchBytes / (kUnitFloats * sizeof(float));

static __device__ __align__(256) float g_attn_scratch[kScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_scratch_ptr[kMaxDevices] = {};  // device address of g_attn_scratch, per device

// Once per device, with that device current: the device address of the array.
cudaError_t scratch_for_current_device(float** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_attn_scratch);
        if (e != cudaSuccess) return e;
        e = tfl::init_attn_decode();  // kernel attributes for this device (no allocation)
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" int tfl_attention_decode_noalloc(tfl_kv* kv, int layer, int pos0, int rows, const void* q, void* out,
                                            void* stream) {
    using namespace tfl;
    char msg[256];
    KvView view;
    int max_pos = 0, n_q = 0, n_kv = 0, layers = 0;
    if (!kv || !q || !out) {
        set_last_error("tfl_attention_decode_noalloc: NULL kv, q or out");
        return TFL_E_ARG;
    }
    if (kv_handle_view(kv, &view, &max_pos, &n_q, &n_kv, &layers) != TFL_OK) return TFL_E_ARG;
    if (layer < 0 || layer >= layers || rows < 1 || rows > kMaxDecodeRows || pos0 < 0 || pos0 + rows > max_pos ||
        ((uintptr_t)q & 15u) || ((uintptr_t)out & 15u)) {
        snprintf(msg, sizeof msg,
                 "tfl_attention_decode_noalloc: layer %d / rows %d / positions %d..%d outside the model or the "
                 "capacity %d, or q/out not 16-byte aligned", layer, rows, pos0, pos0 + rows - 1, max_pos);
        set_last_error(msg);
        return TFL_E_ARG;
    }
    const int nblk = (pos0 + rows - 1) / kAttnUnit + 1;
    const size_t units = (size_t)rows * n_q * nblk;
    if (units > kMaxUnits) {
        snprintf(msg, sizeof msg,
                 "tfl_attention_decode_noalloc: %d rows x %d heads x %d key units of %d positions need %zu "
                 "partials; the fixed scratch holds %zu (16 MiB); use tfl_decode_step or tfl_layer_op instead",
                 rows, n_q, nblk, kAttnUnit, units, kMaxUnits);
        set_last_error(msg);
        return TFL_E_WORKSPACE;
    }
    // the array used is the current device's copy: the cache must live there
    int cur = -1;
    cudaPointerAttributes pa = {};
    cudaError_t e = cudaGetDevice(&cur);
    if (e == cudaSuccess) e = cudaPointerGetAttributes(&pa, view.pages);
    if (e != cudaSuccess) {
        snprintf(msg, sizeof msg, "tfl_attention_decode_noalloc: device query failed: %s", cudaGetErrorString(e));
        set_last_error(msg);
        return TFL_E_CUDA;
    }
    if (pa.type != cudaMemoryTypeDevice || pa.device != cur) {
        snprintf(msg, sizeof msg,
                 "tfl_attention_decode_noalloc: the cache is not device memory of the current device %d (it is on "
                 "device %d); make the model's device current", cur, pa.device);
        set_last_error(msg);
        return TFL_E_ARG;
    }
    float* scratch = nullptr;
    e = scratch_for_current_device(&scratch);
    if (e != cudaSuccess) {
        snprintf(msg, sizeof msg, "tfl_attention_decode_noalloc: scratch set-up failed: %s", cudaGetErrorString(e));
        set_last_error(msg);
        return TFL_E_CUDA;
    }
    AttnDecodeArgs a = {};
    a.q = static_cast<const bf16*>(q);
    a.out = static_cast<bf16*>(out);
    a.pm = scratch;
    a.pl = scratch + units;
    a.po = scratch + 2 * units;
    a.max_blocks = nblk;
    a.n_q = n_q;
    a.n_kv = n_kv;
    a.layer = layer;
    a.rows.n_streams = 1;
    a.rows.n_rows = rows;
    a.rows.row_start[0] = 0;
    a.rows.row_start[1] = rows;
    a.rows.pos0[0] = pos0;
    a.rows.kv[0] = view;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    e = launch_attn_block(a, st, false);
    if (e == cudaSuccess) e = launch_attn_merge(a, st, false);
    if (e != cudaSuccess) {
        snprintf(msg, sizeof msg, "tfl_attention_decode_noalloc: launch failed: %s", cudaGetErrorString(e));
        set_last_error(msg);
        return TFL_E_CUDA;
    }
    set_last_error("");
    return TFL_OK;
}
