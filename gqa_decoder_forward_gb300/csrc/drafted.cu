// Drafted greedy decode: guesses of the next tokens, checked by one causal
// window of the served model, kept up to the first guess that differs from the
// window's own greedy id.  The pages ask that drafted greedy replies equal
// plain greedy ones (issue #1414 "A llama family on Metal: Nanbeige4.3-33B
// served from its bf16 release", reply "Drafting": a smaller Llama on the same
// tokenizer drafting through the lane core's proposer; pull request #1415,
// section "How": the lane host's copy drafts).  Equality holds by construction:
// a window row is bit-identical to a one-row step, and only guesses equal to
// the served model's greedy ids are ever kept.
//
// The host drives the rounds; all arithmetic runs in the decode kernels.  A
// round enqueues the drafter's one-row steps (each step's id comes from the
// previous step's argmax on the device), the served model's window and its
// argmax, then reads the guesses and the window's ids back in one copy.
#include <algorithm>
#include <cstring>
#include <vector>

#include "common.cuh"
#include "tfl.h"

namespace tfl {
int api_fail(int code, const char* msg);
const tfl_config* model_config(const tfl_model* m);
tfl_model* kv_owner(const tfl_kv* kv);
int draft_argmax(tfl_model* m, const void* logits, int n_rows, int32_t* ids, cudaStream_t st);
}  // namespace tfl

namespace {

constexpr int kMaxWindow = 16;   // rows of one stream in one decode step
constexpr int kCopyMaxMatch = 3; // longest suffix a copy draft matches
// Device id slots (int32): the drafter's catch-up tokens end at kPending (the
// pending token), guesses follow it, the window's greedy ids start at kGreedy.
constexpr int kPending = 16;
constexpr int kGreedy = 32;
constexpr int kSlots = 64;
constexpr size_t kSlotBytes = kSlots * sizeof(int32_t);

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

size_t logits_bytes(const tfl_config* c) { return round256((size_t)kMaxWindow * c->vocab * 2); }

int max_draft_len(const tfl_config* c) { return std::min(kMaxWindow, c->max_decode_rows) - 1; }

int copy_draft(const int32_t* t, int n, int max_draft, int32_t* out) {
    for (int m = std::min(kCopyMaxMatch, n - 1); m >= 1; --m) {
        const int32_t* suffix = t + n - m;
        for (int j = n - m - 1; j >= 0; --j) {  // latest earlier occurrence first
            if (!std::equal(suffix, suffix + m, t + j)) continue;
            const int period = n - m - j;  // >= 1
            for (int i = 0; i < max_draft; ++i) out[i] = i < period ? t[n - period + i] : out[i - period];
            return max_draft;
        }
    }
    return 0;
}

#define DCK(call)                                                                   \
    do {                                                                            \
        const cudaError_t e_ = (call);                                              \
        if (e_ != cudaSuccess) return tfl::api_fail(TFL_E_CUDA, cudaGetErrorString(e_)); \
    } while (0)

#define DRUN(call)                 \
    do {                           \
        const int r_ = (call);     \
        if (r_ != TFL_OK) return r_; \
    } while (0)

}  // namespace

extern "C" {

size_t tfl_drafted_workspace_bytes(const tfl_model* target, int draft_len) {
    const tfl_config* c = tfl::model_config(target);
    if (!c || draft_len < 1 || draft_len > max_draft_len(c)) return 0;
    return kSlotBytes + 2 * logits_bytes(c);  // slots, the window's logits, the drafter's logits
}

int tfl_copy_draft(const int32_t* tokens, int n, int max_draft, int32_t* out) {
    if (!tokens || n < 1 || max_draft < 0 || (max_draft > 0 && !out))
        return tfl::api_fail(TFL_E_ARG, "tfl_copy_draft: NULL tokens/out, n < 1 or max_draft < 0");
    return copy_draft(tokens, n, max_draft, out);
}

int tfl_decode_drafted(tfl_model* target, tfl_kv* kv, tfl_model* drafter, tfl_kv* dkv, int draft_len,
                       const int32_t* context, int n_context, int n_tokens, int32_t* out_ids, void* workspace,
                       size_t ws_bytes, tfl_draft_stats* stats, void* stream) {
    using tfl::api_fail;
    const tfl_config* tc = tfl::model_config(target);
    if (!tc || !kv || !context || !out_ids || !workspace)
        return api_fail(TFL_E_ARG, "tfl_decode_drafted: NULL model, cache, context, out_ids or workspace");
    if (tfl::kv_owner(kv) != target) return api_fail(TFL_E_ARG, "tfl_decode_drafted: kv belongs to another model");
    if (n_context < 1 || n_tokens < 1) return api_fail(TFL_E_ARG, "tfl_decode_drafted: n_context or n_tokens < 1");
    if (draft_len < 1 || draft_len > max_draft_len(tc))
        return api_fail(TFL_E_ARG, "tfl_decode_drafted: draft_len outside 1..min(16, max_decode_rows) - 1");
    if (tfl_kv_length(kv) != n_context - 1)
        return api_fail(TFL_E_ARG, "tfl_decode_drafted: length(kv) must be n_context - 1 (the last token is pending)");
    if ((long long)n_context - 1 + n_tokens > tfl_kv_capacity(kv))
        return api_fail(TFL_E_CAPACITY, "tfl_decode_drafted: n_context - 1 + n_tokens exceeds the cache's capacity");
    if (((uintptr_t)workspace & 255u) != 0) return api_fail(TFL_E_ARG, "tfl_decode_drafted: workspace not 256-byte aligned");
    if (ws_bytes < tfl_drafted_workspace_bytes(target, draft_len))
        return api_fail(TFL_E_WORKSPACE, "tfl_decode_drafted: workspace smaller than tfl_drafted_workspace_bytes");
    for (int i = 0; i < n_context; ++i)
        if (context[i] < 0 || context[i] >= tc->vocab)
            return api_fail(TFL_E_ARG, "tfl_decode_drafted: a context id outside [0, vocab)");
    const tfl_config* dc = nullptr;
    int dlen = 0;
    if (drafter) {
        dc = tfl::model_config(drafter);
        if (!dkv || tfl::kv_owner(dkv) != drafter)
            return api_fail(TFL_E_ARG, "tfl_decode_drafted: dkv is NULL or belongs to another model");
        if (drafter == target || dkv == kv)
            return api_fail(TFL_E_ARG, "tfl_decode_drafted: the drafter must be a separate model and cache");
        if (dc->vocab != tc->vocab) return api_fail(TFL_E_ARG, "tfl_decode_drafted: the drafter's vocabulary differs");
        dlen = tfl_kv_length(dkv);
        const int lag = n_context - dlen;
        if (lag < 1 || lag > std::min(kMaxWindow, dc->max_decode_rows))
            return api_fail(TFL_E_ARG, "tfl_decode_drafted: n_context - length(dkv) outside 1..min(16, drafter max_decode_rows)");
        if ((long long)n_context - 1 + n_tokens > tfl_kv_capacity(dkv))
            return api_fail(TFL_E_CAPACITY, "tfl_decode_drafted: n_context - 1 + n_tokens exceeds the drafter cache's capacity");
    }

    cudaStream_t st = (cudaStream_t)stream;
    char* ws = (char*)workspace;
    int32_t* slots = (int32_t*)ws;
    void* tlog = ws + kSlotBytes;
    char* dlog = ws + kSlotBytes + logits_bytes(tc);
    const size_t row_bytes = (size_t)tc->vocab * 2;

    std::vector<int32_t> tok(context, context + n_context);
    tok.reserve((size_t)n_context + n_tokens + kMaxWindow);
    std::vector<int32_t> stage(kMaxWindow), host(kSlots);  // pending + guesses; ids read back
    tfl_draft_stats s;
    std::memset(&s, 0, sizeof s);
    for (int i = 0; i < n_tokens; ++i) out_ids[i] = -1;

    int produced = 0;
    while (produced < n_tokens) {
        const int n_tok = (int)tok.size();        // the last one is pending
        const int k = std::min(draft_len, n_tokens - produced - 1);
        int m = 0;                                // guesses this round
        if (k > 0 && drafter) {
            // catch the drafter up to the pending token (1 or 2 rows after the
            // first round), then k - 1 one-row steps; each argmax feeds the next
            const int lag = n_tok - dlen;
            DCK(cudaMemcpyAsync(slots + kPending - lag + 1, tok.data() + dlen, lag * sizeof(int32_t),
                                cudaMemcpyHostToDevice, st));
            DRUN(tfl_decode_step(drafter, &dkv, 1, slots + kPending - lag + 1, &lag, dlog, stream));
            DRUN(tfl::draft_argmax(drafter, dlog + (size_t)(lag - 1) * row_bytes, 1, slots + kPending + 1, st));
            s.drafter_rows += lag;
            for (int i = 1; i < k; ++i) {
                const int one = 1;
                DRUN(tfl_decode_step(drafter, &dkv, 1, slots + kPending + i, &one, dlog, stream));
                DRUN(tfl::draft_argmax(drafter, dlog, 1, slots + kPending + i + 1, st));
                s.drafter_rows += 1;
            }
            m = k;
        } else {
            stage[0] = tok.back();
            if (k > 0) m = copy_draft(tok.data(), n_tok, k, stage.data() + 1);
            DCK(cudaMemcpyAsync(slots + kPending, stage.data(), (1 + m) * sizeof(int32_t), cudaMemcpyHostToDevice, st));
        }
        const int rows = 1 + m;
        DRUN(tfl_decode_step(target, &kv, 1, slots + kPending, &rows, tlog, stream));
        DRUN(tfl_argmax(target, tlog, rows, slots + kGreedy, stream));
        DCK(cudaMemcpyAsync(host.data() + kPending, slots + kPending, (kGreedy + rows - kPending) * sizeof(int32_t),
                            cudaMemcpyDeviceToHost, st));
        DCK(cudaStreamSynchronize(st));

        int a = 0;  // guesses kept: each equals the greedy id of the row before it
        while (a < m && host[kPending + 1 + a] == host[kGreedy + a]) ++a;
        int take = a + 1;
        int bad = -1;
        for (int i = 0; i < take; ++i)
            if (host[kGreedy + i] < 0) {
                bad = i;
                break;
            }
        if (bad >= 0) take = bad + 1;
        for (int i = 0; i < take; ++i) {
            out_ids[produced + i] = host[kGreedy + i];
            if (i + 1 < take) tok.push_back(host[kGreedy + i]);
        }
        // the served cache keeps the pending token and the kept guesses
        tfl_kv_reset(kv, n_tok + take - 1);
        if (drafter) {
            if (m > 0) dlen = n_tok + std::min(take - 1, m - 1);  // fed: pending, then guesses 1..m-1
            tfl_kv_reset(dkv, std::min(dlen, tfl_kv_length(dkv)));
        }
        s.rounds += 1;
        s.drafted += m;
        s.accepted += take - 1;
        s.target_rows += rows;
        produced += take;
        if (bad >= 0) {
            if (stats) *stats = s;
            return api_fail(TFL_E_NONFINITE, "tfl_decode_drafted: a non-finite logit in the served model's window");
        }
        tok.push_back(host[kGreedy + take - 1]);  // the new pending token
    }
    if (stats) *stats = s;
    return TFL_OK;
}

}  // extern "C"
