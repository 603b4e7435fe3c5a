// The page arena of the C ABI (host only): KV pages handed out lowest id
// first, runs of consecutive pages claimed from the top, both given back
// either at once or once the caller's stream has drained (an event polled,
// never waited on).
#include <algorithm>
#include <map>
#include <mutex>
#include <new>
#include <vector>

#include "pkv_internal.h"

using namespace pkv;

struct pkv_arena {
    pkv_layout layout;
    int32_t page_pos = 0;
    int64_t page_elems = 0;
    int32_t n_pages = 0;
    void *base = nullptr;
    std::vector<uint8_t> taken;  // 1 = a KV page, 2 = a run's page; held or pending release
    std::map<int32_t, int32_t> runs;  // first id -> pages of each run held now
    int32_t n_free = 0;
    int32_t low = 0;  // no free page below this id
    struct Pending {
        void *ev;
        std::vector<int32_t> ids;
    };
    std::vector<Pending> pending;
    pkv_event_ops ops{};
    bool custom_ops = false;
    mutable std::mutex mu;
};

namespace {

int cuda_record(void *, cudaStream_t stream, void **ev) {
    cudaEvent_t e;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return -1;
    if (cudaEventRecord(e, stream) != cudaSuccess) {
        cudaEventDestroy(e);
        return -1;
    }
    *ev = e;
    return 0;
}
int cuda_query(void *, void *ev) {
    cudaError_t r = cudaEventQuery(static_cast<cudaEvent_t>(ev));
    if (r == cudaSuccess) return 0;
    if (r == cudaErrorNotReady) {
        cudaGetLastError();  // not-ready is not sticky; clear it
        return 1;
    }
    return -1;
}
void cuda_destroy(void *, void *ev) { cudaEventDestroy(static_cast<cudaEvent_t>(ev)); }

const pkv_event_ops kCudaOps = {cuda_record, cuda_query, cuda_destroy, nullptr};

void free_page(pkv_arena *a, int32_t id) {
    a->taken[id] = 0;
    a->n_free++;
    if (id < a->low) a->low = id;
}

// Move releases whose stream work has finished back to the free pages.
int poll_pending(pkv_arena *a) {
    int rc = PKV_OK;
    size_t keep = 0;
    for (size_t i = 0; i < a->pending.size(); ++i) {
        auto &p = a->pending[i];
        int q = a->ops.query(a->ops.ctx, p.ev);
        if (q == 0) {
            a->ops.destroy(a->ops.ctx, p.ev);
            for (int32_t id : p.ids) free_page(a, id);
        } else {
            if (q < 0) rc = PKV_ECUDA;
            if (keep != i) a->pending[keep] = std::move(p);
            ++keep;
        }
    }
    a->pending.resize(keep);
    return rc;
}

}  // namespace

extern "C" int pkv_arena_create(const pkv_layout *layout, int32_t page_pos, void *dev_base,
                                size_t bytes, pkv_arena **out) {
    if (!out) return PKV_EINVAL;
    *out = nullptr;
    if (validate_layout(layout) || !page_pos_ok(page_pos) || !dev_base) return PKV_EINVAL;
    if (reinterpret_cast<uintptr_t>(dev_base) & 15u) return PKV_EINVAL;
    int64_t ps = (int64_t)layout->n_layers *
                 layer_elems_f(fp8_of(layout), layout->n_kv_heads, layout->idx_dim, page_pos);
    int64_t n = static_cast<int64_t>(bytes / 2) / ps;
    if (n < 1 || n > INT32_MAX) return PKV_EINVAL;
    pkv_arena *a = new (std::nothrow) pkv_arena;
    if (!a) return PKV_EINVAL;
    a->layout = *layout;
    a->page_pos = page_pos;
    a->page_elems = ps;
    a->n_pages = static_cast<int32_t>(n);
    a->base = dev_base;
    a->taken.assign(static_cast<size_t>(n), 0);
    a->n_free = a->n_pages;
    a->ops = kCudaOps;
    *out = a;
    return PKV_OK;
}

extern "C" int pkv_arena_destroy(pkv_arena *a) {
    if (!a) return PKV_EINVAL;
    for (auto &p : a->pending) a->ops.destroy(a->ops.ctx, p.ev);
    delete a;
    return PKV_OK;
}

extern "C" int pkv_arena_set_event_ops(pkv_arena *a, const pkv_event_ops *ops) {
    if (!a) return PKV_EINVAL;
    std::lock_guard<std::mutex> g(a->mu);
    if (!a->pending.empty()) return PKV_EINVAL;  // events of one kind at a time
    if (ops && (!ops->record || !ops->query || !ops->destroy)) return PKV_EINVAL;
    a->ops = ops ? *ops : kCudaOps;
    a->custom_ops = ops != nullptr;
    return PKV_OK;
}

extern "C" int pkv_arena_info(pkv_arena *a, int32_t *n_pages, int32_t *n_free,
                              int64_t *page_elems) {
    if (!a) return PKV_EINVAL;
    std::lock_guard<std::mutex> g(a->mu);
    int rc = poll_pending(a);
    if (n_pages) *n_pages = a->n_pages;
    if (n_free) *n_free = a->n_free;
    if (page_elems) *page_elems = a->page_elems;
    return rc;
}

extern "C" int pkv_pages_take(pkv_arena *a, int32_t n, int32_t *ids_out) {
    if (!a || n < 0 || (n > 0 && !ids_out)) return PKV_EINVAL;
    std::lock_guard<std::mutex> g(a->mu);
    int rc = poll_pending(a);
    if (rc) return rc;
    if (n > a->n_free) return PKV_EAGAIN;
    int32_t got = 0;
    for (int32_t id = a->low; id < a->n_pages && got < n; ++id) {
        if (!a->taken[id]) {
            a->taken[id] = 1;
            ids_out[got++] = id;
        }
    }
    a->n_free -= got;
    a->low = got ? ids_out[got - 1] + 1 : a->low;
    return PKV_OK;
}

extern "C" int pkv_pages_give(pkv_arena *a, const int32_t *ids, int32_t n, cudaStream_t stream,
                              int32_t defer) {
    if (!a || n < 0 || (n > 0 && !ids)) return PKV_EINVAL;
    std::lock_guard<std::mutex> g(a->mu);
    // every id must be in range, held, and listed once
    std::vector<int32_t> v(ids, ids + n);
    std::sort(v.begin(), v.end());
    for (int32_t i = 0; i < n; ++i) {
        if (v[i] < 0 || v[i] >= a->n_pages || a->taken[v[i]] != 1) return PKV_EINVAL;
        if (i && v[i] == v[i - 1]) return PKV_EINVAL;
    }
    for (auto &p : a->pending)
        for (int32_t id : p.ids)
            if (std::binary_search(v.begin(), v.end(), id)) return PKV_EINVAL;
    if (n == 0) return PKV_OK;
    if (!defer) {
        for (int32_t id : v) free_page(a, id);
        return PKV_OK;
    }
    void *ev = nullptr;
    if (a->ops.record(a->ops.ctx, stream, &ev) != 0) return PKV_ECUDA;
    a->pending.push_back({ev, std::move(v)});
    return PKV_OK;
}

// ---- runs ---------------------------------------------------------------------

extern "C" int pkv_run_pages(const pkv_arena *a, uint64_t run_bytes, int32_t *k_out) {
    if (!a || !k_out) return PKV_EINVAL;
    const uint64_t page_bytes = 2 * static_cast<uint64_t>(a->page_elems);
    const uint64_t k = run_bytes / page_bytes + (run_bytes % page_bytes ? 1 : 0);
    if (k > static_cast<uint64_t>(INT32_MAX)) return PKV_EINVAL;
    *k_out = static_cast<int32_t>(k);
    return PKV_OK;
}

extern "C" int pkv_run_take(pkv_arena *a, int32_t k, int32_t *first_out) {
    if (!a || k < 1 || !first_out) return PKV_EINVAL;
    std::lock_guard<std::mutex> g(a->mu);
    int rc = poll_pending(a);
    if (rc) return rc;
    if (k > a->n_free) return PKV_EAGAIN;
    // scan down from the top; the first window of k free pages met is the
    // highest one
    int32_t streak = 0;
    for (int32_t id = a->n_pages - 1; id >= 0; --id) {
        streak = a->taken[id] ? 0 : streak + 1;
        if (streak == k) {
            for (int32_t j = id; j < id + k; ++j) a->taken[j] = 2;
            a->n_free -= k;
            a->runs[id] = k;
            *first_out = id;
            return PKV_OK;
        }
    }
    return PKV_EAGAIN;
}

namespace {
bool run_held(const pkv_arena *a, int32_t first, int32_t k) {
    auto it = a->runs.find(first);
    return it != a->runs.end() && it->second == k;
}
}  // namespace

extern "C" int pkv_run_give(pkv_arena *a, int32_t first, int32_t k, cudaStream_t stream,
                            int32_t defer) {
    if (!a) return PKV_EINVAL;
    std::lock_guard<std::mutex> g(a->mu);
    if (!run_held(a, first, k)) return PKV_EINVAL;
    std::vector<int32_t> ids(static_cast<size_t>(k));
    for (int32_t j = 0; j < k; ++j) ids[j] = first + j;
    if (defer) {
        void *ev = nullptr;
        if (a->ops.record(a->ops.ctx, stream, &ev) != 0) return PKV_ECUDA;
        a->pending.push_back({ev, std::move(ids)});
    } else {
        for (int32_t id : ids) free_page(a, id);
    }
    a->runs.erase(first);
    return PKV_OK;
}

extern "C" int pkv_run_map(const pkv_arena *a, int32_t first, int32_t k, const uint64_t *part_bytes,
                           int32_t n_parts, uint64_t align, void **ptrs_out) {
    if (!a || n_parts < 0 || (n_parts > 0 && (!part_bytes || !ptrs_out))) return PKV_EINVAL;
    if (align < 16 || align > 4096 || (align & (align - 1))) return PKV_EINVAL;
    std::lock_guard<std::mutex> g(a->mu);
    if (!run_held(a, first, k)) return PKV_EINVAL;
    const uint64_t page_bytes = 2 * static_cast<uint64_t>(a->page_elems);
    const uint64_t lo = reinterpret_cast<uintptr_t>(a->base) + static_cast<uint64_t>(first) * page_bytes;
    const uint64_t hi = lo + static_cast<uint64_t>(k) * page_bytes;
    std::vector<uint64_t> at(static_cast<size_t>(n_parts));
    uint64_t cur = lo;
    for (int32_t i = 0; i < n_parts; ++i) {
        cur = (cur + align - 1) & ~(align - 1);
        if (cur > hi || part_bytes[i] > hi - cur) return PKV_EINVAL;
        at[i] = cur;
        cur += part_bytes[i];
    }
    for (int32_t i = 0; i < n_parts; ++i) ptrs_out[i] = reinterpret_cast<void *>(at[i]);
    return PKV_OK;
}

extern "C" int pkv_arena_pg(const pkv_arena *a, const int32_t *dev_table, int32_t n_table,
                            pkv_pg *out) {
    if (!a || !dev_table || n_table < 1 || !out) return PKV_EINVAL;
    out->base = a->base;
    out->table = dev_table;
    out->page_elems = a->page_elems;
    out->page_pos = a->page_pos;
    out->n_pages = a->n_pages;
    out->n_table = n_table;
    out->reserved = 0;
    return PKV_OK;
}

