// Prompt cache: copying a kept prefix between KV caches, and a host-side index
// of caches by their token prefixes (the prompt cache of the served setup in
// pull request #1415, section "Served": a resumed turn starts from its kept
// prefix).  The copy relies on the caches' identity page tables: the pages of
// one (layer, K or V) are contiguous, so a prefix is one 2-D copy.
#include <cstring>
#include <vector>

#include "common.cuh"
#include "tfl.h"

namespace tfl {
int kv_prefix_geometry(const tfl_kv* kv, const tfl_model* m, bf16** pages, int* n_pages, int* length, int* max_pos);
int kv_set_length(tfl_kv* kv, int length);
int api_fail(int code, const char* msg);
int model_geometry(const tfl_model* m, int* layers, int* n_kv);
}  // namespace tfl

struct tfl_prefix_store {
    struct Entry {
        std::vector<int32_t> tokens;
        tfl_kv* kv;
    };
    int max_entries;
    std::vector<Entry> entries;
};

extern "C" {

int tfl_kv_copy_prefix(tfl_model* m, const tfl_kv* src, tfl_kv* dst, int n, void* stream) {
    using namespace tfl;
    if (!m || !src || !dst) return api_fail(TFL_E_ARG, "tfl_kv_copy_prefix: NULL model or cache");
    bf16 *sp = nullptr, *dp = nullptr;
    int sn = 0, dn = 0, slen = 0, dlen = 0, smax = 0, dmax = 0, layers = 0, n_kv = 0;
    if (kv_prefix_geometry(src, m, &sp, &sn, &slen, &smax) != TFL_OK ||
        kv_prefix_geometry(dst, m, &dp, &dn, &dlen, &dmax) != TFL_OK)
        return api_fail(TFL_E_ARG, "tfl_kv_copy_prefix: a cache of another model");
    if (src == dst) return api_fail(TFL_E_ARG, "tfl_kv_copy_prefix: src and dst are the same cache");
    if (n < 0 || n > slen || n > dmax)
        return api_fail(TFL_E_ARG, "tfl_kv_copy_prefix: n outside 0..min(length(src), capacity(dst))");
    model_geometry(m, &layers, &n_kv);
    if (n > 0) {
        const size_t page_bytes = (size_t)kPage * n_kv * kHeadDim * 2;
        const size_t width = (size_t)((n + kPage - 1) / kPage) * page_bytes;
        const cudaError_t e = cudaMemcpy2DAsync(dp, (size_t)dn * page_bytes, sp, (size_t)sn * page_bytes, width,
                                                (size_t)layers * 2, cudaMemcpyDeviceToDevice, (cudaStream_t)stream);
        if (e != cudaSuccess) return api_fail(TFL_E_CUDA, cudaGetErrorString(e));
    }
    kv_set_length(dst, n);
    return TFL_OK;
}

int tfl_prefix_store_new(int max_entries, tfl_prefix_store** out) {
    if (!out) return tfl::api_fail(TFL_E_ARG, "tfl_prefix_store_new: out is NULL");
    *out = nullptr;
    if (max_entries < 1) return tfl::api_fail(TFL_E_ARG, "tfl_prefix_store_new: max_entries < 1");
    tfl_prefix_store* s = new tfl_prefix_store();
    s->max_entries = max_entries;
    *out = s;
    return TFL_OK;
}

void tfl_prefix_store_free(tfl_prefix_store* s) { delete s; }

int tfl_prefix_store_put(tfl_prefix_store* s, const int32_t* tokens, int n, tfl_kv* kv) {
    if (!s || !tokens || !kv || n < 1) return tfl::api_fail(TFL_E_ARG, "tfl_prefix_store_put: NULL argument or n < 1");
    if ((int)s->entries.size() >= s->max_entries)
        return tfl::api_fail(TFL_E_CAPACITY, "tfl_prefix_store_put: the store is full (remove an entry first)");
    tfl_prefix_store::Entry e;
    e.tokens.assign(tokens, tokens + n);
    e.kv = kv;
    s->entries.push_back(std::move(e));
    return TFL_OK;
}

int tfl_prefix_store_match(tfl_prefix_store* s, const int32_t* tokens, int n, tfl_kv** kv, int* matched) {
    if (!s || (!tokens && n > 0) || n < 0 || !kv || !matched)
        return tfl::api_fail(TFL_E_ARG, "tfl_prefix_store_match: NULL argument or n < 0");
    *kv = nullptr;
    *matched = 0;
    for (const tfl_prefix_store::Entry& e : s->entries) {
        const int lim = std::min(n, (int)e.tokens.size());
        int c = 0;
        while (c < lim && e.tokens[c] == tokens[c]) ++c;
        if (c > 0 && c >= *matched) {
            *matched = c;
            *kv = e.kv;
        }
    }
    return TFL_OK;
}

int tfl_prefix_store_remove(tfl_prefix_store* s, const tfl_kv* kv) {
    if (!s) return tfl::api_fail(TFL_E_ARG, "tfl_prefix_store_remove: NULL store");
    std::vector<tfl_prefix_store::Entry> keep;
    for (tfl_prefix_store::Entry& e : s->entries)
        if (e.kv != kv) keep.push_back(std::move(e));
    s->entries.swap(keep);
    return TFL_OK;
}

int tfl_prefix_store_size(const tfl_prefix_store* s) { return s ? (int)s->entries.size() : -1; }

}  // extern "C"
