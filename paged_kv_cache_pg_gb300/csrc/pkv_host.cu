// Host side of the C ABI: argument checks, host pg_at, tensor maps, and the
// entry points that pack kernel parameters and launch.
#include <algorithm>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <vector>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "pkv_internal.h"

namespace pkv {

int launch_status(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ECUDA; }

int validate_layout(const pkv_layout *L) {
    if (!L) return PKV_EINVAL;
    if (L->n_layers < 1 || L->n_kv_heads < 1 || L->n_kv_heads > 64) return PKV_EINVAL;
    if (L->head_dim != kHeadDim) return PKV_EINVAL;
    if (L->idx_dim != 0 && L->idx_dim != kIdxDim) return PKV_EINVAL;
    if (L->kv_format != PKV_KV_BF16 && L->kv_format != PKV_KV_E4M3) return PKV_EINVAL;
    return PKV_OK;
}


int sm_count(int *out) {
    static std::atomic<int> cached[64];  // per device, 0 until first asked
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ECUDA;
    if (dev < 0 || dev >= 64) return PKV_ECUDA;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return PKV_ECUDA;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    *out = n;
    return PKV_OK;
}

// Check one stream's descriptor against the layout.
static int validate_pg(const pkv_layout *L, const pkv_pg &pg) {
    if (!pg.base || (reinterpret_cast<uintptr_t>(pg.base) & 15u)) return PKV_EINVAL;
    if (!page_pos_ok(pg.page_pos)) return PKV_EINVAL;
    int64_t want =
        (int64_t)L->n_layers * layer_elems_f(fp8_of(L), L->n_kv_heads, L->idx_dim, pg.page_pos);
    if (pg.page_elems != want) return PKV_EINVAL;
    if (pg.table) {
        if (pg.n_pages < 1 || pg.n_table < 1) return PKV_EINVAL;
    }
    return PKV_OK;
}

static int64_t capacity(const pkv_pg &pg) {
    return pg.table ? (int64_t)pg.n_table * pg.page_pos : pg.page_pos;
}

int fill_common(const pkv_layout *L, const pkv_seq *seqs, int32_t n_seqs, int32_t layer,
                int32_t n_q_heads, int32_t *dev_status, Common *c) {
    int rc = validate_layout(L);
    if (rc) return rc;
    if (n_seqs < 0 || n_seqs > PKV_MAX_SEQS || (n_seqs > 0 && !seqs)) return PKV_EINVAL;
    if (layer < 0 || layer >= L->n_layers) return PKV_EINVAL;
    if (n_q_heads < 1 || n_q_heads % L->n_kv_heads != 0) return PKV_EINVAL;
    std::memset(c, 0, sizeof(*c));
    c->n_seqs = n_seqs;
    c->n_kv_heads = L->n_kv_heads;
    c->idx_dim = L->idx_dim;
    c->layer = layer;
    c->n_q_heads = n_q_heads;
    c->group = n_q_heads / L->n_kv_heads;
    c->kv_fp8 = fp8_of(L);
    c->status = reinterpret_cast<uint32_t *>(dev_status);
    int32_t tok = 0;
    for (int32_t s = 0; s < n_seqs; ++s) {
        const pkv_seq &q = seqs[s];
        rc = validate_pg(L, q.pg);
        if (rc) return rc;
        if (q.len < 0 || q.n_new < 0 || q.n_new > q.len || q.len > capacity(q.pg))
            return PKV_EINVAL;
        SeqDev &d = c->seq[s];
        const uint16_t *base = static_cast<const uint16_t *>(q.pg.base);
        d.layer_base = base + (int64_t)layer * layer_elems_f(fp8_of(L), L->n_kv_heads,
                                                             L->idx_dim, q.pg.page_pos);
        d.table = q.pg.table;
        d.ps = q.pg.page_elems;
        d.ptok = q.pg.page_pos;
        d.n_pages = q.pg.table ? q.pg.n_pages : 1;
        d.n_table = q.pg.table ? q.pg.n_table : 1;
        d.len = q.len;
        d.n_new = q.n_new;
        d.tok_off = tok;
        if ((int64_t)tok + q.n_new > INT32_MAX / 2) return PKV_EINVAL;
        tok += q.n_new;
    }
    return PKV_OK;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---- TMA row maps ------------------------------------------------------------

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        cudaGetLastError();
    });
    return fn;
}

namespace {
struct MapKey {
    uintptr_t base;
    uint64_t rows;
    bool bytes8;
    bool tile;
    int box_rows, box_chunks;
};
std::mutex g_map_mu;
std::vector<std::pair<MapKey, RowMap>> g_maps;  // encoded maps, most recent last
}  // namespace

int row_map(DecodeMaps &maps, int &n_maps, const void *base, uint64_t rows, bool bytes8,
            bool tile, int box_rows, int box_chunks) {
    if (rows == 0 || rows > (1ull << 31) || !aligned16(base)) return -1;
    if (tile ? (bytes8 || (box_rows != 64 && box_rows != 128) || (box_chunks != 2 && box_chunks != 4))
             : (box_rows != 16 || box_chunks != 1))
        return -1;
    RowMap m;
    bool have = false;
    {
        std::lock_guard<std::mutex> g(g_map_mu);
        for (auto &e : g_maps)
            if (e.first.base == reinterpret_cast<uintptr_t>(base) && e.first.rows == rows &&
                e.first.bytes8 == bytes8 && e.first.tile == tile && e.first.box_rows == box_rows &&
                e.first.box_chunks == box_chunks) {
                m = e.second;
                have = true;
                break;
            }
    }
    if (!have) {
        auto fn = encode_fn();
        if (!fn) return -1;
        // bf16 rows: 256 elements (512 B), boxes of 64 x 16; e4m3 code rows:
        // 256 bytes, boxes of 128 x 16 (both 128-byte inner boxes).  The tile
        // view: dims {64, rows, 4 column chunks}, strides 512 B (a row) and
        // 128 B (a chunk), boxes of {64, box_rows, box_chunks}.
        cuuint64_t dims[3] = {256, rows, 1};
        cuuint64_t strides[2] = {bytes8 ? 256u : 512u, 0};
        cuuint32_t box[3] = {bytes8 ? 128u : 64u, 16, 1};
        if (tile) {
            dims[0] = 64;
            dims[2] = 4;
            strides[1] = 128;
            box[1] = static_cast<cuuint32_t>(box_rows);
            box[2] = static_cast<cuuint32_t>(box_chunks);
        }
        cuuint32_t estr[3] = {1, 1, 1};
        CUresult r = fn(reinterpret_cast<CUtensorMap *>(m.bytes),
                        bytes8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        tile ? 3 : 2, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return -1;
        std::lock_guard<std::mutex> g(g_map_mu);
        if (g_maps.size() >= 256) g_maps.erase(g_maps.begin());
        g_maps.push_back({{reinterpret_cast<uintptr_t>(base), rows, bytes8, tile, box_rows, box_chunks}, m});
    }
    for (int i = 0; i < n_maps; ++i)
        if (std::memcmp(maps.map[i].bytes, m.bytes, sizeof(m.bytes)) == 0) return i;
    if (n_maps >= kMaxMaps) return -1;
    maps.map[n_maps] = m;
    return n_maps++;
}

void plan_maps(Common &c, const pkv_layout *L, const pkv_seq *seqs, DecodeMaps &maps, bool tiles) {
    int n_maps = 0;
    for (int s = 0; s < c.n_seqs; ++s) {
        SeqDev &d = c.seq[s];
        d.tma = -1;
        d.tma_k = d.tma_v = -1;
        const pkv_pg &pg = seqs[s].pg;
        const int64_t layer_off =
            (int64_t)c.layer * layer_elems_f(fp8_of(L), L->n_kv_heads, L->idx_dim, pg.page_pos);
        if (fp8_of(L)) {
            // e4m3 code rows of 256 bytes: whole 16-row runs by TMA when every
            // page and this layer's block start on a 256-byte row
            const int64_t page_bytes = 2 * pg.page_elems, layer_bytes = 2 * layer_off;
            if (pg.page_pos % 16 != 0 || page_bytes % 256 != 0 || layer_bytes % 256 != 0) continue;
            const uint64_t rows = (uint64_t)(pg.table ? pg.n_pages : 1) * page_bytes / 256;
            d.tma = row_map(maps, n_maps, pg.base, rows, true);
            d.layer_row = layer_bytes / 256;
            d.page_rows = page_bytes / 256;
            continue;
        }
        if (pg.page_pos % 16 != 0 || pg.page_elems % 256 != 0 || layer_off % 256 != 0) continue;
        const uint64_t rows = (uint64_t)(pg.table ? pg.n_pages : 1) * pg.page_elems / 256;
        d.tma = row_map(maps, n_maps, pg.base, rows, false);
        d.layer_row = layer_off / 256;
        d.page_rows = pg.page_elems / 256;
        // a chunk kernel's K slot (a 128-key tile over 128 dims) and V slot
        // (64 keys over 256 dims) start on multiples of their key counts, so
        // in pages of a multiple of those counts each is one run: one copy.
        // (A decode tile stays four 2D copies of 16 rows: one 3D copy of its
        // 8 KB made the decode chain about 3 % slower, its rows arriving later.)
        if (tiles && d.tma >= 0) {
            if (pg.page_pos % 128 == 0)
                d.tma_k = static_cast<int16_t>(row_map(maps, n_maps, pg.base, rows, false, true, 128, 2));
            if (pg.page_pos % 64 == 0)
                d.tma_v = static_cast<int16_t>(row_map(maps, n_maps, pg.base, rows, false, true, 64, 4));
        }
    }
}

static int total_new(const Common &c) {
    int t = 0;
    for (int s = 0; s < c.n_seqs; ++s) t += c.seq[s].n_new;
    return t;
}

}  // namespace pkv

using namespace pkv;

// ============================================================================
// layout and host pg_at
// ============================================================================

extern "C" int pkv_layout_page_elems(const pkv_layout *layout, int32_t page_pos, int64_t *out) {
    if (validate_layout(layout) || !page_pos_ok(page_pos) || !out) return PKV_EINVAL;
    *out = (int64_t)layout->n_layers *
           layer_elems_f(fp8_of(layout), layout->n_kv_heads, layout->idx_dim, page_pos);
    return PKV_OK;
}

extern "C" int pkv_pg_row(const pkv_layout *L, const pkv_pg *pg, const int32_t *host_table,
                          int32_t layer, int32_t kind, int32_t head, int32_t pos, int64_t *out) {
    if (validate_layout(L) || !pg || !out || validate_pg(L, *pg)) return PKV_EINVAL;
    if (layer < 0 || layer >= L->n_layers || pos < 0) return PKV_EINVAL;
    const bool fp8 = fp8_of(L);
    if (kind < PKV_K || kind > (fp8 ? PKV_VS : PKV_P)) return PKV_EINVAL;
    const bool per_head = kind == PKV_K || kind == PKV_V || kind == PKV_KS || kind == PKV_VS;
    if (per_head && (head < 0 || head >= L->n_kv_heads)) return PKV_EINVAL;
    if ((kind == PKV_IK || kind == PKV_P) && L->idx_dim == 0) return PKV_EINVAL;
    if (pg->table && !host_table) return PKV_EINVAL;
    const int32_t ptok = pg->page_pos;
    const int64_t position = kind == PKV_P ? 4 * (int64_t)pos : pos;
    if (position >= capacity(*pg)) return PKV_EINVAL;
    int64_t page_off = 0;
    int32_t row = static_cast<int32_t>(position);
    if (pg->table) {
        int32_t page = static_cast<int32_t>(position / ptok);
        int32_t id = host_table[page];
        if (id < 0 || id >= pg->n_pages) return PKV_EINVAL;
        page_off = (int64_t)id * pg->page_elems;
        row = static_cast<int32_t>(position % ptok);
    }
    int64_t in_layer;
    const int32_t H = L->n_kv_heads;
    if (fp8) {
        // byte offsets for every kind of an e4m3 layout
        switch (kind) {
        case PKV_K: in_layer = off8_code(false, H, ptok, head, row); break;
        case PKV_V: in_layer = off8_code(true, H, ptok, head, row); break;
        case PKV_KS: in_layer = off8_scale(false, H, ptok, head, row); break;
        case PKV_VS: in_layer = off8_scale(true, H, ptok, head, row); break;
        case PKV_IK: in_layer = 2 * off_ik_f(true, H, L->idx_dim, ptok, row); break;
        default: in_layer = 2 * off_p_f(true, H, L->idx_dim, ptok, row / 4); break;
        }
        *out = 2 * page_off + 2 * (int64_t)layer * layer_elems_f(true, H, L->idx_dim, ptok) + in_layer;
        return PKV_OK;
    }
    switch (kind) {
    case PKV_K: in_layer = off_k(ptok, head, row); break;
    case PKV_V: in_layer = off_v(H, ptok, head, row); break;
    case PKV_IK: in_layer = off_ik(H, L->idx_dim, ptok, row); break;
    default: in_layer = off_p(H, L->idx_dim, ptok, row / 4); break;
    }
    *out = page_off + (int64_t)layer * layer_elems(H, L->idx_dim, ptok) + in_layer;
    return PKV_OK;
}

// ============================================================================
// kernel entry points
// ============================================================================

extern "C" int pkv_store(const pkv_layout *L, const pkv_seq *seqs, int32_t n_seqs, int32_t layer,
                         const void *k_new, const void *v_new, const void *ik_new,
                         int32_t *dev_status, cudaStream_t stream) {
    Common c;
    int rc = fill_common(L, seqs, n_seqs, layer, L ? L->n_kv_heads : 1, dev_status, &c);
    if (rc) return rc;
    int tok = total_new(c);
    if (tok == 0) return PKV_OK;
    if (!k_new || !v_new || (L->idx_dim && !ik_new)) return PKV_EINVAL;
    if (!aligned16(k_new) || !aligned16(v_new) || (L->idx_dim && !aligned16(ik_new)))
        return PKV_EINVAL;
    auto launch = c.kv_fp8 ? launch_store8 : launch_store;
    return launch(c, tok, static_cast<const uint16_t *>(k_new), static_cast<const uint16_t *>(v_new),
                  static_cast<const uint16_t *>(ik_new), stream);
}

extern "C" int pkv_gather(const pkv_layout *L, const pkv_seq *seqs, int32_t n_seqs, int32_t layer,
                          int32_t kind, void *out, int32_t *dev_status, cudaStream_t stream) {
    Common c;
    int rc = fill_common(L, seqs, n_seqs, layer, L ? L->n_kv_heads : 1, dev_status, &c);
    if (rc) return rc;
    if (kind < PKV_K || kind > (c.kv_fp8 ? PKV_VS : PKV_P)) return PKV_EINVAL;
    if ((kind == PKV_IK || kind == PKV_P) && L->idx_dim == 0) return PKV_EINVAL;
    int64_t rows = 0;
    for (int s = 0; s < c.n_seqs; ++s) {
        c.seq[s].work_off = static_cast<int32_t>(rows);
        rows += kind == PKV_P ? c.seq[s].len / 4 : c.seq[s].len;
    }
    if (rows == 0) return PKV_OK;
    if (!out || !aligned16(out) || rows > INT32_MAX / 2) return PKV_EINVAL;
    if (c.kv_fp8 && kind != PKV_IK && kind != PKV_P)  // codes or scales
        return launch_gather8(c, kind, rows, out, stream);
    return launch_gather(c, kind, rows, static_cast<uint16_t *>(out), stream);
}

extern "C" int pkv_pool(const pkv_layout *L, const pkv_seq *seqs, int32_t n_seqs, int32_t layer,
                        int32_t *dev_status, cudaStream_t stream) {
    Common c;
    int rc = fill_common(L, seqs, n_seqs, layer, L ? L->n_kv_heads : 1, dev_status, &c);
    if (rc) return rc;
    if (L->idx_dim == 0) return PKV_EINVAL;
    int32_t blocks = 0;
    for (int s = 0; s < c.n_seqs; ++s) {
        SeqDev &d = c.seq[s];
        d.work_off = blocks;
        blocks += d.len / 4 - (d.len - d.n_new) / 4;
    }
    if (blocks == 0) return PKV_OK;
    return launch_pool(c, blocks, stream);
}

// Dense bf16 decode calls with a unit of more than 16 query columns (a
// stream's draft window: 4 queries x 8 heads) run on the tensor-core chunk
// kernel: the MMA work per key is large enough there that tcgen05 beats the
// warp-MMA decode (the window's new rows are stored first when the call
// brings them).
static bool tensor_route(const Common &c, bool sparse) {
    if (sparse || c.kv_fp8) return false;
    for (int s = 0; s < c.n_seqs; ++s)
        if (c.seq[s].n_new * c.group > 16) return true;
    return false;
}

static int decode_common(const pkv_layout *L, const pkv_seq *seqs, int32_t n_seqs,
                         int32_t layer, int32_t n_q_heads, bool sparse, int32_t k,
                         int32_t *dev_status, Common *c, DecodePlan *plan, bool *tensor = nullptr) {
    int rc = fill_common(L, seqs, n_seqs, layer, n_q_heads, dev_status, c);
    if (rc) return rc;
    if (sparse) {
        if (k < 1 || k > 256) return PKV_EINVAL;
        for (int s = 0; s < c->n_seqs; ++s)
            if (c->seq[s].n_new != 1) return PKV_EINVAL;
    } else {
        for (int s = 0; s < c->n_seqs; ++s)
            if (c->seq[s].n_new * c->group > 32) return PKV_EINVAL;  // query columns of a unit
    }
    int nsm = 0;
    rc = sm_count(&nsm);
    if (rc) return rc;
    const bool route = tensor_route(*c, sparse);
    if (tensor) *tensor = route;
    return route ? plan_prefill(*c, nsm, plan) : plan_decode(*c, sparse, k, nsm, plan);
}

// The tensor-core route of a dense decode call: the chunk kernel attends the
// window, reading the new rows (when given) from the inputs and storing them
// into their pages itself; its split partials are merged by the decode
// combine.
static int launch_tensor_route(const pkv_layout *L, const pkv_seq *seqs, const Common &c,
                               const DecodePlan &plan, const void *q, const void *k_new,
                               const void *v_new, const void *ik_new, void *out, float *ws,
                               cudaStream_t stream) {
    DecodeMaps maps;
    Common cc = c;
    plan_maps(cc, L, seqs, maps, true);
    return launch_prefill(cc, plan, maps, static_cast<const uint16_t *>(q),
                          static_cast<uint16_t *>(out), ws, static_cast<const uint16_t *>(k_new),
                          static_cast<const uint16_t *>(v_new), static_cast<const uint16_t *>(ik_new),
                          stream);
}

extern "C" int pkv_decode_ws_size(const pkv_layout *L, const pkv_seq *seqs, int32_t n_seqs,
                                  int32_t n_q_heads, size_t *bytes) {
    if (!bytes) return PKV_EINVAL;
    Common c;
    DecodePlan plan;
    int rc = decode_common(L, seqs, n_seqs, 0, n_q_heads, false, 0, nullptr, &c, &plan);
    if (rc) return rc;
    *bytes = plan.ws_bytes;
    return PKV_OK;
}

extern "C" int pkv_decode(const pkv_layout *L, const pkv_seq *seqs, int32_t n_seqs, int32_t layer,
                          int32_t n_q_heads, const void *q, const void *k_new, const void *v_new,
                          const void *ik_new, void *out, void *ws, size_t ws_bytes,
                          int32_t *dev_status, cudaStream_t stream) {
    Common c;
    DecodePlan plan;
    bool tensor = false;
    int rc = decode_common(L, seqs, n_seqs, layer, n_q_heads, false, 0, dev_status, &c, &plan, &tensor);
    if (rc) return rc;
    if (plan.total_items == 0) return PKV_OK;
    if (!q || !out || !aligned16(q) || !aligned16(out)) return PKV_EINVAL;
    if ((k_new == nullptr) != (v_new == nullptr)) return PKV_EINVAL;
    if (k_new) {
        if (!aligned16(k_new) || !aligned16(v_new)) return PKV_EINVAL;
        if (L->idx_dim && (!ik_new || !aligned16(ik_new))) return PKV_EINVAL;
    }
    if (plan.ws_bytes > 0 &&
        (!ws || ws_bytes < plan.ws_bytes || (reinterpret_cast<uintptr_t>(ws) & 255u)))
        return PKV_EINVAL;
    if (tensor)
        return launch_tensor_route(L, seqs, c, plan, q, k_new, v_new, L->idx_dim ? ik_new : nullptr,
                                   out, static_cast<float *>(ws), stream);
    DecodeMaps maps;  // copied into the launch's parameters
    plan_maps(c, L, seqs, maps, false);
    if (c.kv_fp8)
        return launch_decode8(c, plan, maps, static_cast<const uint16_t *>(q),
                              static_cast<uint16_t *>(out), static_cast<float *>(ws),
                              static_cast<const uint16_t *>(k_new),
                              static_cast<const uint16_t *>(v_new),
                              k_new ? static_cast<const uint16_t *>(ik_new) : nullptr, stream);
    return launch_decode(c, plan, maps, false, static_cast<const uint16_t *>(q), nullptr, 0,
                         static_cast<uint16_t *>(out), static_cast<float *>(ws),
                         static_cast<const uint16_t *>(k_new), static_cast<const uint16_t *>(v_new),
                         k_new ? static_cast<const uint16_t *>(ik_new) : nullptr, stream);
}

extern "C" int pkv_decode_static(const pkv_layout *L, const pkv_seq *seqs, int32_t n_seqs,
                                 int32_t layer, int32_t n_q_heads, const void *q,
                                 const void *k_new, const void *v_new, const void *ik_new,
                                 void *out, int32_t *dev_status, cudaStream_t stream) {
    Common c;
    DecodePlan plan;
    bool tensor = false;
    int rc = decode_common(L, seqs, n_seqs, layer, n_q_heads, false, 0, dev_status, &c, &plan, &tensor);
    if (rc) return rc;
    if (plan.ws_bytes > kStaticScratchBytes) return PKV_EINVAL;  // over the fixed scratch
    if (plan.total_items == 0) return PKV_OK;
    if (!q || !out || !aligned16(q) || !aligned16(out)) return PKV_EINVAL;
    if ((k_new == nullptr) != (v_new == nullptr)) return PKV_EINVAL;
    if (k_new) {
        if (!aligned16(k_new) || !aligned16(v_new)) return PKV_EINVAL;
        if (L->idx_dim && (!ik_new || !aligned16(ik_new))) return PKV_EINVAL;
    }
    void *scratch = nullptr;
    rc = static_scratch(&scratch);
    if (rc) return rc;
    if (tensor)
        return launch_tensor_route(L, seqs, c, plan, q, k_new, v_new, L->idx_dim ? ik_new : nullptr,
                                   out, static_cast<float *>(scratch), stream);
    DecodeMaps maps;
    plan_maps(c, L, seqs, maps, false);
    if (c.kv_fp8)
        return launch_decode8(c, plan, maps, static_cast<const uint16_t *>(q),
                              static_cast<uint16_t *>(out), static_cast<float *>(scratch),
                              static_cast<const uint16_t *>(k_new),
                              static_cast<const uint16_t *>(v_new),
                              k_new ? static_cast<const uint16_t *>(ik_new) : nullptr, stream);
    return launch_decode(c, plan, maps, false, static_cast<const uint16_t *>(q), nullptr, 0,
                         static_cast<uint16_t *>(out), static_cast<float *>(scratch),
                         static_cast<const uint16_t *>(k_new), static_cast<const uint16_t *>(v_new),
                         k_new ? static_cast<const uint16_t *>(ik_new) : nullptr, stream);
}

extern "C" int pkv_sparse_ws_size(const pkv_layout *L, const pkv_seq *seqs, int32_t n_seqs,
                                  int32_t n_q_heads, int32_t k, size_t *bytes) {
    if (!bytes) return PKV_EINVAL;
    Common c;
    DecodePlan plan;
    int rc = decode_common(L, seqs, n_seqs, 0, n_q_heads, true, k, nullptr, &c, &plan);
    if (rc) return rc;
    *bytes = plan.ws_bytes;
    return PKV_OK;
}

extern "C" int pkv_sparse_decode(const pkv_layout *L, const pkv_seq *seqs, int32_t n_seqs,
                                 int32_t layer, int32_t n_q_heads, const void *q,
                                 const int32_t *ids, int32_t k, void *out, void *ws,
                                 size_t ws_bytes, int32_t *dev_status, cudaStream_t stream) {
    Common c;
    DecodePlan plan;
    int rc = decode_common(L, seqs, n_seqs, layer, n_q_heads, true, k, dev_status, &c, &plan);
    if (rc) return rc;
    if (c.kv_fp8) return PKV_EINVAL;
    if (plan.total_items == 0) return PKV_OK;
    if (!q || !out || !ids || !aligned16(q) || !aligned16(out)) return PKV_EINVAL;
    if (plan.ws_bytes > 0 &&
        (!ws || ws_bytes < plan.ws_bytes || (reinterpret_cast<uintptr_t>(ws) & 255u)))
        return PKV_EINVAL;
    for (int s = 0; s < c.n_seqs; ++s) {  // selected blocks: cp.async path
        c.seq[s].tma = -1;
        c.seq[s].tma_k = c.seq[s].tma_v = -1;
    }
    DecodeMaps maps;
    return launch_decode(c, plan, maps, true, static_cast<const uint16_t *>(q), ids, k,
                         static_cast<uint16_t *>(out), static_cast<float *>(ws), nullptr, nullptr,
                         nullptr, stream);
}

static int prefill_common(const pkv_layout *L, const pkv_seq *seqs, int32_t n_seqs, int32_t layer,
                          int32_t n_q_heads, int32_t *dev_status, Common *c, DecodePlan *plan) {
    int rc = fill_common(L, seqs, n_seqs, layer, n_q_heads, dev_status, c);
    if (rc) return rc;
    if (c->kv_fp8) return PKV_EINVAL;  // the tensor-core prefill reads bf16 rows
    int nsm = 0;
    rc = sm_count(&nsm);
    if (rc) return rc;
    return plan_prefill(*c, nsm, plan);
}

extern "C" int pkv_prefill_ws_size(const pkv_layout *L, const pkv_seq *seqs, int32_t n_seqs,
                                   int32_t n_q_heads, size_t *bytes) {
    if (!bytes) return PKV_EINVAL;
    Common c;
    DecodePlan plan;
    int rc = prefill_common(L, seqs, n_seqs, 0, n_q_heads, nullptr, &c, &plan);
    if (rc) return rc;
    *bytes = plan.ws_bytes;
    return PKV_OK;
}

extern "C" int pkv_prefill(const pkv_layout *L, const pkv_seq *seqs, int32_t n_seqs, int32_t layer,
                           int32_t n_q_heads, const void *q, void *out, void *ws, size_t ws_bytes,
                           int32_t *dev_status, cudaStream_t stream) {
    Common c;
    DecodePlan plan;
    int rc = prefill_common(L, seqs, n_seqs, layer, n_q_heads, dev_status, &c, &plan);
    if (rc) return rc;
    if (plan.total_items == 0) return PKV_OK;
    if (!q || !out || !aligned16(q) || !aligned16(out)) return PKV_EINVAL;
    if (plan.ws_bytes > 0 &&
        (!ws || ws_bytes < plan.ws_bytes || (reinterpret_cast<uintptr_t>(ws) & 255u)))
        return PKV_EINVAL;
    DecodeMaps maps;
    plan_maps(c, L, seqs, maps, true);
    return launch_prefill(c, plan, maps, static_cast<const uint16_t *>(q),
                          static_cast<uint16_t *>(out), static_cast<float *>(ws), nullptr, nullptr,
                          nullptr, stream);
}

extern "C" int pkv_block_scores(const pkv_layout *L, const pkv_seq *seqs, int32_t n_seqs,
                                int32_t layer, int32_t n_q_heads, const void *qi, float *scores,
                                int32_t ld, int32_t *dev_status, cudaStream_t stream) {
    Common c;
    int rc = fill_common(L, seqs, n_seqs, layer, n_q_heads, dev_status, &c);
    if (rc) return rc;
    if (L->idx_dim == 0) return PKV_EINVAL;
    int32_t max_nb = 0;
    for (int s = 0; s < c.n_seqs; ++s) {
        if (c.seq[s].n_new != 1) return PKV_EINVAL;
        max_nb = std::max(max_nb, c.seq[s].len / 4);
    }
    if (ld < max_nb || ld < 0) return PKV_EINVAL;
    if (c.n_seqs == 0 || ld == 0) return PKV_OK;
    if (!qi || !scores || !aligned16(qi)) return PKV_EINVAL;
    return launch_scores(c, scores, ld, static_cast<const uint16_t *>(qi), max_nb, stream);
}

extern "C" int pkv_topk(const pkv_seq *seqs, int32_t n_seqs, int32_t n_q_heads,
                        const float *scores, int32_t ld, int32_t k, int32_t *ids,
                        cudaStream_t stream) {
    if (n_seqs < 0 || n_seqs > PKV_MAX_SEQS || (n_seqs > 0 && !seqs)) return PKV_EINVAL;
    if (n_q_heads < 1 || k < 1 || k > 256) return PKV_EINVAL;
    Common c;
    std::memset(&c, 0, sizeof(c));
    c.n_seqs = n_seqs;
    c.n_q_heads = n_q_heads;
    for (int s = 0; s < n_seqs; ++s) {
        if (seqs[s].len < 0) return PKV_EINVAL;
        if (seqs[s].len / 4 > ld) return PKV_EINVAL;
        c.seq[s].len = seqs[s].len;
    }
    if (n_seqs == 0) return PKV_OK;
    if (!scores || !ids || ld < 0) return PKV_EINVAL;
    return launch_topk(c, scores, ld, k, ids, stream);
}
