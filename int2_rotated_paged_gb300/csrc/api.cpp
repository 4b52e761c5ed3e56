// api.cpp -- host side of the C ABI: argument checks, the cache handle, the host free
// list of the page table, and the launches.  No device memory is allocated here.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <vector>

#include "../../include/oscar_kv.h"
#include "internal.h"

using namespace oscar;

struct oscar_cache {
    oscar_cache_desc d;
    uint8_t* pool;
    uint16_t* bf16;
    int32_t* pt;
    int32_t* lens_dev;
    uint32_t* vmax_dev;                       // [batch][hkv] after the lengths (vmax_offset)
    std::vector<int64_t> len;                 // tokens held per request
    std::vector<std::vector<int32_t>> rows;   // physical pages held per request
    std::vector<int32_t> free_list;           // popped from the back
    std::vector<int32_t> dirty_lo;            // first row entry not yet on the device
    std::vector<char> vmax_stale;             // the request's value-scale maxima need zeroing
    bool clear_device;                        // the device table / lengths need zeroing
    bool lens_dirty;
    int32_t g;
    PageFmt fmt;                              // byte layout of a (page, KV head) block
    // optional per-launch timing of the decode kernel: event pairs, filled in launch order
    std::vector<cudaEvent_t> timing_ev;
    int32_t timing_used = 0;
};

static void free_timing(oscar_cache* c) {
    for (cudaEvent_t e : c->timing_ev) cudaEventDestroy(e);
    c->timing_ev.clear();
    c->timing_used = 0;
}

namespace {

std::atomic<int> g_last_cuda{0};
std::atomic<int64_t> g_launches{0};

int cuda_fail(cudaError_t e) {
    g_last_cuda = (int)e;
    return OSCAR_ECUDA;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

bool desc_ok(const oscar_cache_desc* d) {
    if (!d) return false;
    if (d->batch < 1 || d->batch > kMaxBatch) return false;
    if (d->num_kv_heads < 1 || d->num_q_heads < 1) return false;
    if (d->num_q_heads % d->num_kv_heads) return false;
    const int g = d->num_q_heads / d->num_kv_heads;
    if (g > kMaxG || (g > 8 && g != 12 && g != 16)) return false;
    if (d->head_dim != kD || d->page_size != kPage) return false;
    if (d->group_size != 64 && d->group_size != 128) return false;
    if (d->group_size_v != 0 && d->group_size_v != 64 && d->group_size_v != 128) return false;
    if (d->sink != kSink || d->window != kWindow) return false;
    if (d->max_pages_total < 1 || d->max_pages_per_seq < 1) return false;
    if (!(d->clip_k > 0.f && d->clip_k <= 1.f && d->clip_v > 0.f && d->clip_v <= 1.f)) return false;
    return true;
}

cudaStream_t S(void* s) { return (cudaStream_t)s; }

PageFmt fmt_of(const oscar_cache_desc* d) {
    return page_fmt(d->group_size, d->group_size_v ? d->group_size_v : d->group_size);
}

// Pages the INT2 history of a request needs once it holds `len` tokens.
int64_t pages_for(int64_t len) {
    int64_t t = len > kSlots ? len - kSlots : 0;
    return (t + kPage - 1) / kPage;
}

int take_pages(oscar_cache* c, int32_t b, int64_t new_len) {
    int64_t need = pages_for(new_len);
    int64_t have = (int64_t)c->rows[b].size();
    if (need <= have) return OSCAR_OK;
    if (need > c->d.max_pages_per_seq) return OSCAR_ENOPAGES;
    if (need - have > (int64_t)c->free_list.size()) return OSCAR_ENOPAGES;
    for (int64_t i = have; i < need; ++i) {
        c->rows[b].push_back(c->free_list.back());
        c->free_list.pop_back();
    }
    c->dirty_lo[b] = std::min<int32_t>(c->dirty_lo[b], (int32_t)have);
    return OSCAR_OK;
}

int sync(oscar_cache* c, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    if (c->clear_device) {
        e = cudaMemsetAsync(c->pt, 0, oscar_page_table_bytes(&c->d), s);
        if (e == cudaSuccess) e = cudaMemsetAsync(c->lens_dev, 0, oscar_seq_lens_bytes(&c->d), s);
        if (e != cudaSuccess) return cuda_fail(e);
        c->clear_device = false;
        c->lens_dirty = true;
        std::fill(c->vmax_stale.begin(), c->vmax_stale.end(), 0);
    }
    for (int32_t b = 0; b < c->d.batch; ++b) {
        if (!c->vmax_stale[b]) continue;
        e = cudaMemsetAsync(c->vmax_dev + (size_t)b * c->d.num_kv_heads, 0, sizeof(uint32_t) * c->d.num_kv_heads, s);
        if (e != cudaSuccess) return cuda_fail(e);
        c->vmax_stale[b] = 0;
    }
    for (int32_t b = 0; b < c->d.batch; ++b) {
        const int32_t lo = c->dirty_lo[b];
        const int32_t hi = (int32_t)c->rows[b].size();
        if (lo < hi) {
            e = cudaMemcpyAsync(c->pt + (size_t)b * c->d.max_pages_per_seq + lo, c->rows[b].data() + lo,
                                sizeof(int32_t) * (hi - lo), cudaMemcpyHostToDevice, s);
            if (e != cudaSuccess) return cuda_fail(e);
        }
        c->dirty_lo[b] = INT32_MAX;
    }
    if (c->lens_dirty) {
        std::vector<int32_t> l(c->len.begin(), c->len.end());
        e = cudaMemcpyAsync(c->lens_dev, l.data(), sizeof(int32_t) * l.size(), cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e);
        c->lens_dirty = false;
    }
    return OSCAR_OK;
}

}  // namespace

namespace oscar {
void count_launches(int n) { g_launches += n; }
}  // namespace oscar

extern "C" {

void oscar_default_desc(oscar_cache_desc* d) {
    if (!d) return;
    std::memset(d, 0, sizeof(*d));
    d->batch = 1;
    d->num_kv_heads = 1;
    d->num_q_heads = 1;
    d->head_dim = kD;
    d->page_size = kPage;
    d->group_size = kGroup;
    d->group_size_v = kGroup;
    d->sink = kSink;
    d->window = kWindow;
    d->max_pages_total = 1;
    d->max_pages_per_seq = 1;
    d->clip_k = 0.96f;
    d->clip_v = 0.92f;
}

size_t oscar_page_head_bytes(const oscar_cache_desc* d) {
    if (!desc_ok(d)) return 0;
    return (size_t)fmt_of(d).bytes;
}
size_t oscar_pool_bytes(const oscar_cache_desc* d) {
    if (!desc_ok(d)) return 0;
    return (size_t)d->max_pages_total * d->num_kv_heads * fmt_of(d).bytes;
}
size_t oscar_bf16_bytes(const oscar_cache_desc* d) {
    if (!desc_ok(d)) return 0;
    return (size_t)d->batch * d->num_kv_heads * 2 * kSlots * kD * sizeof(uint16_t);
}
size_t oscar_page_table_bytes(const oscar_cache_desc* d) {
    if (!desc_ok(d)) return 0;
    return (size_t)d->batch * d->max_pages_per_seq * sizeof(int32_t);
}
size_t oscar_seq_lens_bytes(const oscar_cache_desc* d) {
    if (!desc_ok(d)) return 0;
    return (vmax_offset(d->batch) + (size_t)d->batch * d->num_kv_heads * sizeof(uint32_t) + 15) / 16 * 16;
}

int oscar_cache_create(const oscar_cache_desc* d, void* pool, void* bf16, int32_t* page_table,
                       int32_t* seq_lens, oscar_cache** out) {
    if (!out) return OSCAR_EINVAL;
    *out = nullptr;
    if (!desc_ok(d) || !pool || !bf16 || !page_table || !seq_lens) return OSCAR_EINVAL;
    if (!aligned16(pool) || !aligned16(bf16) || !aligned16(page_table) || !aligned16(seq_lens))
        return OSCAR_EALIGN;
    oscar_cache* c = new oscar_cache();
    c->d = *d;
    if (!c->d.group_size_v) c->d.group_size_v = c->d.group_size;
    c->fmt = fmt_of(&c->d);
    c->pool = (uint8_t*)pool;
    c->bf16 = (uint16_t*)bf16;
    c->pt = page_table;
    c->lens_dev = seq_lens;
    c->vmax_dev = (uint32_t*)((uint8_t*)seq_lens + vmax_offset(d->batch));
    c->vmax_stale.assign(d->batch, 0);
    c->len.assign(d->batch, 0);
    c->rows.assign(d->batch, {});
    c->g = d->num_q_heads / d->num_kv_heads;
    c->free_list.resize(d->max_pages_total);
    for (int32_t i = 0; i < d->max_pages_total; ++i) c->free_list[i] = d->max_pages_total - 1 - i;
    c->dirty_lo.assign(d->batch, INT32_MAX);
    c->clear_device = true;
    c->lens_dirty = true;
    *out = c;
    return OSCAR_OK;
}

int oscar_cache_destroy(oscar_cache* c) {
    if (c) free_timing(c);
    delete c;
    return OSCAR_OK;
}

int64_t oscar_cache_length(const oscar_cache* c, int32_t b) {
    if (!c) return OSCAR_EINVAL;
    if (b < 0 || b >= c->d.batch) return OSCAR_ERANGE;
    return c->len[b];
}

// ------------------------------------------------------------------ kv_page_table

int kv_page_table_init(oscar_cache* c, const int32_t* page_order) {
    if (!c) return OSCAR_EINVAL;
    const int32_t n = c->d.max_pages_total;
    std::vector<int32_t> order(n);
    if (page_order) {
        std::vector<char> seen(n, 0);
        for (int32_t i = 0; i < n; ++i) {
            int32_t p = page_order[i];
            if (p < 0 || p >= n || seen[p]) return OSCAR_EINVAL;
            seen[p] = 1;
            order[i] = p;
        }
    } else {
        for (int32_t i = 0; i < n; ++i) order[i] = i;
    }
    c->free_list.assign(order.rbegin(), order.rend());
    for (auto& r : c->rows) r.clear();
    std::fill(c->len.begin(), c->len.end(), 0);
    std::fill(c->dirty_lo.begin(), c->dirty_lo.end(), INT32_MAX);
    c->clear_device = true;
    return OSCAR_OK;
}

int kv_page_table_reserve(oscar_cache* c, int32_t b, int64_t new_len) {
    if (!c) return OSCAR_EINVAL;
    if (b < 0 || b >= c->d.batch || new_len < 0) return OSCAR_ERANGE;
    return take_pages(c, b, new_len);
}

int kv_page_table_release(oscar_cache* c, int32_t b) {
    if (!c) return OSCAR_EINVAL;
    if (b < 0 || b >= c->d.batch) return OSCAR_ERANGE;
    auto& r = c->rows[b];
    for (auto it = r.rbegin(); it != r.rend(); ++it) c->free_list.push_back(*it);
    r.clear();
    c->dirty_lo[b] = INT32_MAX;
    c->len[b] = 0;
    c->lens_dirty = true;
    c->vmax_stale[b] = 1;
    return OSCAR_OK;
}

int kv_page_table_sync(oscar_cache* c, void* stream) {
    if (!c) return OSCAR_EINVAL;
    return sync(c, S(stream));
}

int kv_page_table_read(const oscar_cache* c, int32_t b, int32_t* pages, int32_t max_out) {
    if (!c) return OSCAR_EINVAL;
    if (b < 0 || b >= c->d.batch) return OSCAR_ERANGE;
    const auto& r = c->rows[b];
    if (pages)
        for (int32_t i = 0; i < max_out && i < (int32_t)r.size(); ++i) pages[i] = r[i];
    return (int)r.size();
}

int32_t kv_page_table_free_pages(const oscar_cache* c) {
    return c ? (int32_t)c->free_list.size() : OSCAR_EINVAL;
}

// ------------------------------------------------------------------ write path

// Host part of an append: argument and capacity checks, page reservation, page-table upload and
// the kernel parameters.  *any = false when no token is appended.  c->len is left to the caller.
static int prepare_append(oscar_cache* c, const void* k, const void* v, const int32_t* new_tokens,
                          const float* rk, cudaStream_t s, AppendParams& p, bool* any) {
    *any = false;
    if (!c || !new_tokens) return OSCAR_EINVAL;
    const oscar_cache_desc& d = c->d;
    int64_t rows = 0;
    int64_t need_pages = 0;
    for (int32_t b = 0; b < d.batch; ++b) {
        if (new_tokens[b] < 0) return OSCAR_EINVAL;
        int64_t l1 = c->len[b] + new_tokens[b];
        if (l1 > INT32_MAX / 2) return OSCAR_ERANGE;
        int64_t p = pages_for(l1);
        if (p > d.max_pages_per_seq) return OSCAR_ENOPAGES;
        need_pages += std::max<int64_t>(0, p - (int64_t)c->rows[b].size());
        rows += new_tokens[b];
    }
    if (rows == 0) return OSCAR_OK;
    if (!k || !v || !rk) return OSCAR_EINVAL;
    if (!aligned16(k) || !aligned16(v) || !aligned16(rk)) return OSCAR_EALIGN;
    if (need_pages > (int64_t)c->free_list.size()) return OSCAR_ENOPAGES;

    for (int32_t b = 0; b < d.batch; ++b) {
        int rc = take_pages(c, b, c->len[b] + new_tokens[b]);
        if (rc != OSCAR_OK) return rc;   // cannot happen after the capacity check above
    }
    int rc = sync(c, s);
    if (rc != OSCAR_OK) return rc;
    std::memset(&p, 0, sizeof(p));
    p.fmt = c->fmt;
    p.batch = d.batch;
    p.hkv = d.num_kv_heads;
    p.clip_k = d.clip_k;
    p.clip_v = d.clip_v;
    p.k = (const uint16_t*)k;
    p.v = (const uint16_t*)v;
    p.rk = rk;
    p.pool = c->pool;
    p.bf16 = c->bf16;
    p.page_table = c->pt;
    p.seq_lens = c->lens_dev;
    p.vmax = c->vmax_dev;
    p.max_pps = d.max_pages_per_seq;
    int64_t off = 0;
    int32_t jobs = 0;
    for (int32_t b = 0; b < d.batch; ++b) {
        AppendReq& r = p.req[b];
        r.len0 = (int32_t)c->len[b];
        r.n_new = new_tokens[b];
        r.tok_off = off;
        int32_t l1 = r.len0 + r.n_new;
        r.e0 = std::max<int32_t>(kSink, r.len0 - kWindow);
        r.e1 = std::max<int32_t>(kSink, l1 - kWindow);
        r.job0 = jobs;
        r.page0 = (r.e0 - kSink) / kPage;
        if (r.e1 > r.e0) jobs += (r.e1 - 1 - kSink) / kPage - r.page0 + 1;
        off += new_tokens[b];
    }
    p.n_jobs = jobs;
    *any = true;
    return OSCAR_OK;
}

int kv_quant_append(oscar_cache* c, const void* k, const void* v, const int32_t* new_tokens,
                    const float* rk, void* stream) {
    AppendParams p;
    bool any = false;
    int rc = prepare_append(c, k, v, new_tokens, rk, S(stream), p, &any);
    if (rc != OSCAR_OK || !any) return rc;
    cudaError_t e = launch_append(p, S(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    for (int32_t b = 0; b < c->d.batch; ++b) c->len[b] += new_tokens[b];
    return OSCAR_OK;
}

size_t kv_quant_append_layers_workspace_bytes(int32_t n_layers) {
    if (n_layers < 1 || n_layers > kMaxAppendLayers) return 0;
    return ((size_t)n_layers * sizeof(AppendParams) + 255) / 256 * 256;
}

int kv_quant_append_layers(oscar_cache* const* caches, int32_t n_layers, const void* const* k, const void* const* v,
                           const int32_t* new_tokens, const float* const* rk, void* workspace, size_t workspace_bytes,
                           void* stream) {
    if (!caches || !k || !v || !rk || !new_tokens || n_layers < 1 || n_layers > kMaxAppendLayers) return OSCAR_EINVAL;
    const oscar_cache* c0 = caches[0];
    if (!c0) return OSCAR_EINVAL;
    for (int32_t l = 0; l < n_layers; ++l) {
        const oscar_cache* c = caches[l];
        if (!c || c->d.batch != c0->d.batch || c->d.num_kv_heads != c0->d.num_kv_heads ||
            c->fmt.gk != c0->fmt.gk || c->fmt.gv != c0->fmt.gv || c->len != c0->len)
            return OSCAR_EINVAL;
        for (int32_t j = 0; j < l; ++j)
            if (caches[j] == c) return OSCAR_EINVAL;   // a cache twice would append twice
    }
    if (!workspace || workspace_bytes < kv_quant_append_layers_workspace_bytes(n_layers)) return OSCAR_EWORKSPACE;
    if (!aligned16(workspace)) return OSCAR_EALIGN;
    const cudaStream_t s = S(stream);
    std::vector<AppendParams> ps(n_layers);
    for (int32_t l = 0; l < n_layers; ++l) {
        bool any = false;
        int rc = prepare_append(caches[l], k[l], v[l], new_tokens, rk[l], s, ps[l], &any);
        if (rc != OSCAR_OK) return rc;
        if (!any) return OSCAR_OK;   // no token for any request (the same for every layer)
    }
    cudaError_t e = cudaMemcpyAsync(workspace, ps.data(), sizeof(AppendParams) * n_layers, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e);
    e = launch_append_layers((const AppendParams*)workspace, ps[0], n_layers, s);
    if (e != cudaSuccess) return cuda_fail(e);
    for (int32_t l = 0; l < n_layers; ++l)
        for (int32_t b = 0; b < caches[l]->d.batch; ++b) caches[l]->len[b] += new_tokens[b];
    return OSCAR_OK;
}

// ------------------------------------------------------------------ read path

// request slots of a decode call: slot b is request b with its one query (identity mapping)
static void identity_slots(DecodeParams& p) {
    p.g_real = p.g;
    p.qpr = 1;
    for (int32_t b = 0; b < p.batch; ++b) {
        p.row[b] = b;
        p.q0[b] = b;
        p.nq[b] = 1;
        p.lim[b] = INT32_MAX;
    }
}

static const int kMaxSplits = 64;   // SIMT path: INT2 splits + 1 BF16 split per (request, KV head)
static std::atomic<int> g_decode_path{OSCAR_PATH_WARP_MMA};
static constexpr int kDefaultWaitIters = 2000;   // about 2 s
static std::atomic<int> g_wait_iters{kDefaultWaitIters};
static std::atomic<int> g_wait_probe{0};

static int pick_pps(const oscar_cache* c) {
    int64_t total = 0;
    int64_t longest = 0;
    for (int32_t b = 0; b < c->d.batch; ++b) {
        total += pages_for(c->len[b]);
        longest = std::max<int64_t>(longest, pages_for(c->len[b]));
    }
    total *= c->d.num_kv_heads;
    // about 8 split CTAs per SM of a 152-SM part, at least 4 pages (256 tokens) each
    int64_t pps = std::max<int64_t>(4, (total + 152 * 8 - 1) / (152 * 8));
    pps = std::max<int64_t>(pps, (longest + kMaxSplits - 2) / (kMaxSplits - 1));
    return (int)pps;
}

static int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (!cached[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached[dev] = n;
    }
    return cached[dev];
}

// Page-streaming units (warps) of the warp-MMA kernel: one CTA per SM (fewer when there are few pages).
static int mma_unit_count(int32_t g, int64_t pages, int32_t* n_units) {
    const int sms = sm_count();
    if (sms <= 0) return cuda_fail(cudaGetLastError());
    const int per = mma_units_per_cta(g);
    const int64_t ctas = std::min<int64_t>(std::min(sms, kMaxMmaUnits / per), (pages + per - 1) / per);
    *n_units = (int32_t)(ctas * per);
    return OSCAR_OK;
}

struct WsLayout {
    size_t qrot, simt, mma, bf16, err, total;
};

// Workspace layouts: the error word first (offset 0 in every layout, so one status query serves
// decode and prefill workspaces alike), then the rotated queries and the split-K partials.
static WsLayout ws_layout(const oscar_cache* c) {
    const size_t per = (size_t)c->g * (2 + kD) * sizeof(float);
    const size_t bh = (size_t)c->d.batch * c->d.num_kv_heads;
    WsLayout w;
    w.err = 0;
    w.qrot = 256;
    w.simt = w.qrot + (size_t)c->d.batch * c->d.num_q_heads * kD * sizeof(float);
    w.mma = w.simt + bh * kMaxSplits * per;
    w.bf16 = w.mma + (bh + kMaxMmaUnits) * per;   // one slot per (request, KV head) run of a unit
    w.total = w.bf16 + bh * per;
    return w;
}

size_t oscar_decode_workspace_bytes(const oscar_cache* c) {
    if (!c) return 0;
    return ws_layout(c).total;
}

int oscar_set_decode_path(int32_t path) {
    if (path != OSCAR_PATH_SIMT && path != OSCAR_PATH_WARP_MMA) return OSCAR_EINVAL;
    g_decode_path = path;
    return OSCAR_OK;
}

int oscar_set_wait_limit(int32_t iters) {
    if (iters < 0) {
        g_wait_iters = kDefaultWaitIters;
        return OSCAR_OK;
    }
    if (iters > 1000000) return OSCAR_EINVAL;
    g_wait_iters = iters;
    return OSCAR_OK;
}

int oscar_set_wait_probe(int32_t on) {
    g_wait_probe = on ? 1 : 0;
    return OSCAR_OK;
}

int oscar_decode_status(const void* workspace, size_t workspace_bytes, const oscar_cache* c, void* stream) {
    if (!c || !workspace) return OSCAR_EINVAL;
    const WsLayout w = ws_layout(c);
    if (workspace_bytes < w.err + sizeof(int32_t)) return OSCAR_EWORKSPACE;
    int32_t err = 0;
    cudaError_t e = cudaMemcpyAsync(&err, (const uint8_t*)workspace + w.err, sizeof(err), cudaMemcpyDeviceToHost,
                                    S(stream));
    if (e == cudaSuccess) e = cudaStreamSynchronize(S(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    return err ? OSCAR_ETIMEOUT : OSCAR_OK;
}

static int check_decode_args(const oscar_cache* c, const void* q, int32_t q_dtype, const float* rk,
                             const void* out, int32_t out_dtype, const void* workspace, size_t workspace_bytes) {
    if (!c || !q || !rk || !out) return OSCAR_EINVAL;
    if ((q_dtype != OSCAR_DTYPE_F32 && q_dtype != OSCAR_DTYPE_BF16) ||
        (out_dtype != OSCAR_DTYPE_F32 && out_dtype != OSCAR_DTYPE_BF16))
        return OSCAR_EINVAL;
    if (!workspace || workspace_bytes < oscar_decode_workspace_bytes(c)) return OSCAR_EWORKSPACE;
    if (!aligned16(q) || !aligned16(rk) || !aligned16(out) || !aligned16(workspace)) return OSCAR_EALIGN;
    return OSCAR_OK;
}

// Kernel parameters of a decode call over the cache's current lengths (page table uploaded first).
static int prepare_decode(oscar_cache* c, const void* q, int32_t q_dtype, const float* rk, void* out,
                          int32_t out_dtype, void* workspace, cudaStream_t s, DecodeParams& p) {
    int rc = sync(c, s);
    if (rc != OSCAR_OK) return rc;
    std::memset(&p, 0, sizeof(p));
    p.fmt = c->fmt;
    p.batch = c->d.batch;
    p.hkv = c->d.num_kv_heads;
    p.g = c->g;
    p.pps = pick_pps(c);
    p.max_splits = kMaxSplits;
    p.q = q;
    p.q_dtype = q_dtype;
    p.rk = rk;
    p.out = out;
    p.out_dtype = out_dtype;
    p.pool = c->pool;
    p.bf16 = c->bf16;
    p.page_table = c->pt;
    p.max_pps = c->d.max_pages_per_seq;
    const WsLayout w = ws_layout(c);
    uint8_t* ws = (uint8_t*)workspace;
    p.qrot = (float*)(ws + w.qrot);
    p.partial = (float*)(ws + w.simt);
    p.part_mma = (float*)(ws + w.mma);
    p.part_bf16 = (float*)(ws + w.bf16);
    p.err = (int32_t*)(ws + w.err);
    p.vmax = c->vmax_dev;
    p.path = g_decode_path;
    p.wait_iters = g_wait_iters;
    p.wait_probe = g_wait_probe;
    int64_t pages = 0;
    for (int32_t b = 0; b < c->d.batch; ++b) {
        p.len[b] = (int32_t)c->len[b];
        p.page_off[b] = (int32_t)pages;
        pages += (int64_t)int2_pages(p.len[b]) * c->d.num_kv_heads;
    }
    p.page_off[c->d.batch] = (int32_t)pages;
    if (pages > INT32_MAX / 4) return OSCAR_ERANGE;
    p.total_pages = (int32_t)pages;
    identity_slots(p);
    if (p.path == OSCAR_PATH_WARP_MMA && pages > 0) {
        rc = mma_unit_count(c->g, pages, &p.n_units);
        if (rc != OSCAR_OK) return rc;
    }
    return OSCAR_OK;
}

static cudaEvent_t* next_timing(oscar_cache* c) {
    if (c->timing_used * 2 + 1 >= (int32_t)c->timing_ev.size()) return nullptr;
    cudaEvent_t* t = &c->timing_ev[2 * c->timing_used];
    ++c->timing_used;
    return t;
}

int oscar_decode_attention(oscar_cache* c, const void* q, int32_t q_dtype, const float* rk,
                           void* out, int32_t out_dtype, void* workspace, size_t workspace_bytes,
                           void* stream) {
    int rc = check_decode_args(c, q, q_dtype, rk, out, out_dtype, workspace, workspace_bytes);
    if (rc != OSCAR_OK) return rc;
    DecodeParams p;
    rc = prepare_decode(c, q, q_dtype, rk, out, out_dtype, workspace, S(stream), p);
    if (rc != OSCAR_OK) return rc;
    cudaError_t e = launch_decode(p, S(stream), next_timing(c));
    return e == cudaSuccess ? OSCAR_OK : cuda_fail(e);
}

int oscar_decode_step(oscar_cache* c, const void* k, const void* v, const void* q, int32_t q_dtype,
                      const float* rk, void* out, int32_t out_dtype, void* workspace, size_t workspace_bytes,
                      void* stream) {
    int rc = check_decode_args(c, q, q_dtype, rk, out, out_dtype, workspace, workspace_bytes);
    if (rc != OSCAR_OK) return rc;
    const std::vector<int32_t> ones(c->d.batch, 1);
    if (g_decode_path != OSCAR_PATH_WARP_MMA) {
        rc = kv_quant_append(c, k, v, ones.data(), rk, stream);
        if (rc != OSCAR_OK) return rc;
        return oscar_decode_attention(c, q, q_dtype, rk, out, out_dtype, workspace, workspace_bytes, stream);
    }
    // the lengths after the append must fit the page-offset arithmetic before anything changes
    int64_t pages = 0;
    for (int32_t b = 0; b < c->d.batch; ++b) pages += (int64_t)int2_pages((int32_t)c->len[b] + 1) * c->d.num_kv_heads;
    if (pages > INT32_MAX / 4) return OSCAR_ERANGE;
    AppendParams a;
    bool any = false;
    rc = prepare_append(c, k, v, ones.data(), rk, S(stream), a, &any);
    if (rc != OSCAR_OK) return rc;
    for (int32_t b = 0; b < c->d.batch; ++b) c->len[b] += 1;
    DecodeParams p;
    rc = prepare_decode(c, q, q_dtype, rk, out, out_dtype, workspace, S(stream), p);
    if (rc != OSCAR_OK) return rc;
    cudaError_t e = launch_decode_step(p, a, S(stream), next_timing(c));
    return e == cudaSuccess ? OSCAR_OK : cuda_fail(e);
}

// Device staging of oscar_decode_step_host: keys, values, queries, output (256-byte aligned parts).
struct StepStaging {
    size_t kv_bytes, q_bytes, out_bytes;
    size_t k, v, q, out, total;
};
static StepStaging step_staging(const oscar_cache* c, int32_t q_dtype, int32_t out_dtype) {
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    StepStaging st;
    st.kv_bytes = (size_t)c->d.batch * c->d.num_kv_heads * kD * sizeof(uint16_t);
    st.q_bytes = (size_t)c->d.batch * c->d.num_q_heads * kD * (q_dtype == OSCAR_DTYPE_BF16 ? 2 : 4);
    st.out_bytes = (size_t)c->d.batch * c->d.num_q_heads * kD * (out_dtype == OSCAR_DTYPE_BF16 ? 2 : 4);
    st.k = 0;
    st.v = up(st.kv_bytes);
    st.q = st.v + up(st.kv_bytes);
    st.out = st.q + up(st.q_bytes);
    st.total = st.out + up(st.out_bytes);
    return st;
}

size_t oscar_decode_step_host_staging_bytes(const oscar_cache* c, int32_t q_dtype, int32_t out_dtype) {
    if (!c || (q_dtype != OSCAR_DTYPE_F32 && q_dtype != OSCAR_DTYPE_BF16) ||
        (out_dtype != OSCAR_DTYPE_F32 && out_dtype != OSCAR_DTYPE_BF16))
        return 0;
    return step_staging(c, q_dtype, out_dtype).total;
}

int oscar_decode_step_host(oscar_cache* c, const void* k_host, const void* v_host, const void* q_host, int32_t q_dtype,
                           const float* rk, void* out_host, int32_t out_dtype, void* staging, size_t staging_bytes,
                           void* workspace, size_t workspace_bytes, void* stream) {
    if (!c || !k_host || !v_host || !q_host || !out_host) return OSCAR_EINVAL;
    const size_t need = oscar_decode_step_host_staging_bytes(c, q_dtype, out_dtype);
    if (need == 0) return OSCAR_EINVAL;
    if (!staging || staging_bytes < need) return OSCAR_EWORKSPACE;
    if (!aligned16(staging)) return OSCAR_EALIGN;
    const StepStaging st = step_staging(c, q_dtype, out_dtype);
    uint8_t* sb = (uint8_t*)staging;
    int rc = check_decode_args(c, sb + st.q, q_dtype, rk, sb + st.out, out_dtype, workspace, workspace_bytes);
    if (rc != OSCAR_OK) return rc;
    const cudaStream_t s = S(stream);
    cudaError_t e = cudaMemcpyAsync(sb + st.k, k_host, st.kv_bytes, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(sb + st.v, v_host, st.kv_bytes, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(sb + st.q, q_host, st.q_bytes, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e);
    rc = oscar_decode_step(c, sb + st.k, sb + st.v, sb + st.q, q_dtype, rk, sb + st.out, out_dtype, workspace,
                           workspace_bytes, stream);
    if (rc != OSCAR_OK) return rc;
    e = cudaMemcpyAsync(out_host, sb + st.out, st.out_bytes, cudaMemcpyDeviceToHost, s);
    return e == cudaSuccess ? OSCAR_OK : cuda_fail(e);
}

int oscar_kernel_timing(oscar_cache* c, int32_t capacity) {
    if (!c || capacity < 0 || capacity > (1 << 20)) return OSCAR_EINVAL;
    free_timing(c);
    c->timing_ev.resize((size_t)capacity * 2, nullptr);
    for (auto& ev : c->timing_ev) {
        cudaError_t e = cudaEventCreate(&ev);
        if (e != cudaSuccess) {
            ev = nullptr;
            free_timing(c);
            return cuda_fail(e);
        }
    }
    return OSCAR_OK;
}

int oscar_kernel_timing_read(oscar_cache* c, float* ms, int32_t max_n, int32_t* n_out) {
    if (!c || !n_out || max_n < 0 || (max_n > 0 && !ms)) return OSCAR_EINVAL;
    const int32_t n = std::min(max_n, c->timing_used);
    for (int32_t i = 0; i < n; ++i) {
        cudaError_t e = cudaEventSynchronize(c->timing_ev[2 * i + 1]);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms[i], c->timing_ev[2 * i], c->timing_ev[2 * i + 1]);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    *n_out = n;
    c->timing_used = 0;
    return OSCAR_OK;
}

// ------------------------------------------------------------------ chunked prefill attention

// Query tokens per request slot: the most that keep qpr * G a head count the kernels take
// (1..8, 12, 16), so that one unpacked page serves several queries.
static int prefill_qpr(int g) {
    for (int k = 16 / g; k > 1; --k) {
        const int gv = k * g;
        if (gv <= 8 || gv == 12 || gv == 16) return k;
    }
    return 1;
}

static WsLayout prefill_ws_layout(const oscar_cache* c) {
    const int gv = c->g * prefill_qpr(c->g);
    const size_t per = (size_t)gv * (2 + kD) * sizeof(float);
    const size_t bh = (size_t)kMaxBatch * c->d.num_kv_heads;
    WsLayout w;
    w.err = 0;
    w.qrot = 256;
    w.simt = w.qrot + (size_t)kMaxBatch * c->d.num_kv_heads * gv * kD * sizeof(float);
    w.mma = w.simt;                                 // no SIMT partials on this path
    w.bf16 = w.mma + (bh + kMaxMmaUnits) * per;
    w.total = w.bf16 + bh * per;
    return w;
}

size_t oscar_prefill_workspace_bytes(const oscar_cache* c) {
    if (!c) return 0;
    return prefill_ws_layout(c).total;
}

int oscar_prefill_attention(oscar_cache* c, const void* q, int32_t q_dtype, const int32_t* n_q, const float* rk,
                            void* out, int32_t out_dtype, void* workspace, size_t workspace_bytes, void* stream) {
    if (!c || !n_q) return OSCAR_EINVAL;
    if (g_decode_path != OSCAR_PATH_WARP_MMA) return OSCAR_EINVAL;
    int64_t rows = 0;
    for (int32_t b = 0; b < c->d.batch; ++b) {
        if (n_q[b] < 0 || n_q[b] > kWindow || n_q[b] > c->len[b]) return OSCAR_ERANGE;
        rows += n_q[b];
    }
    if (rows == 0) return OSCAR_OK;
    if (!q || !rk || !out) return OSCAR_EINVAL;
    if ((q_dtype != OSCAR_DTYPE_F32 && q_dtype != OSCAR_DTYPE_BF16) ||
        (out_dtype != OSCAR_DTYPE_F32 && out_dtype != OSCAR_DTYPE_BF16))
        return OSCAR_EINVAL;
    const WsLayout w = prefill_ws_layout(c);
    if (!workspace || workspace_bytes < w.total) return OSCAR_EWORKSPACE;
    if (!aligned16(q) || !aligned16(rk) || !aligned16(out) || !aligned16(workspace)) return OSCAR_EALIGN;
    int rc = sync(c, S(stream));
    if (rc != OSCAR_OK) return rc;
    const int qpr = prefill_qpr(c->g);
    uint8_t* ws = (uint8_t*)workspace;
    // request slots: runs of qpr consecutive chunk queries of one request, launched 256 slots at a time
    struct Slot {
        int32_t row, q0, nq, lim;
    };
    std::vector<Slot> slots;
    int64_t qrow = 0;
    for (int32_t b = 0; b < c->d.batch; ++b) {
        const int64_t first = c->len[b] - n_q[b];     // position of the chunk's first token
        for (int32_t i = 0; i < n_q[b]; i += qpr)
            slots.push_back({b, (int32_t)(qrow + i), std::min(qpr, n_q[b] - i), (int32_t)(first + i)});
        qrow += n_q[b];
    }
    for (size_t s0 = 0; s0 < slots.size(); s0 += kMaxBatch) {
        const int32_t nb = (int32_t)std::min<size_t>(kMaxBatch, slots.size() - s0);
        DecodeParams p;
        std::memset(&p, 0, sizeof(p));
        p.fmt = c->fmt;
        p.batch = nb;
        p.hkv = c->d.num_kv_heads;
        p.g = c->g * qpr;
        p.g_real = c->g;
        p.qpr = qpr;
        p.pps = 4;
        p.max_splits = kMaxSplits;
        p.q = q;
        p.q_dtype = q_dtype;
        p.rk = rk;
        p.out = out;
        p.out_dtype = out_dtype;
        p.pool = c->pool;
        p.bf16 = c->bf16;
        p.page_table = c->pt;
        p.max_pps = c->d.max_pages_per_seq;
        p.qrot = (float*)(ws + w.qrot);
        p.partial = nullptr;
        p.part_mma = (float*)(ws + w.mma);
        p.part_bf16 = (float*)(ws + w.bf16);
        p.err = (int32_t*)(ws + w.err);
        p.vmax = c->vmax_dev;
        p.path = OSCAR_PATH_WARP_MMA;
        p.wait_iters = g_wait_iters;
        p.wait_probe = g_wait_probe;
        int64_t pages = 0;
        for (int32_t v = 0; v < nb; ++v) {
            const Slot& sl = slots[s0 + v];
            p.len[v] = (int32_t)c->len[sl.row];
            p.row[v] = sl.row;
            p.q0[v] = sl.q0;
            p.nq[v] = sl.nq;
            p.lim[v] = sl.lim;
            p.page_off[v] = (int32_t)pages;
            pages += (int64_t)int2_pages(p.len[v]) * c->d.num_kv_heads;
        }
        p.page_off[nb] = (int32_t)pages;
        if (pages > INT32_MAX / 4) return OSCAR_ERANGE;
        p.total_pages = (int32_t)pages;
        if (pages > 0) {
            rc = mma_unit_count(p.g, pages, &p.n_units);
            if (rc != OSCAR_OK) return rc;
        }
        cudaError_t e = launch_decode(p, S(stream));
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return OSCAR_OK;
}

// ------------------------------------------------------------------ calibration

size_t oscar_build_rk_workspace_bytes(int32_t num_kv_heads) {
    return num_kv_heads > 0 ? build_rk_ws_bytes(num_kv_heads) : 0;
}

int oscar_build_rk(const float* q, int64_t n, int32_t num_kv_heads, float* rk, void* workspace,
                   size_t workspace_bytes, void* stream) {
    if (!q || !rk || n < 1 || num_kv_heads < 1) return OSCAR_EINVAL;
    if (!workspace || workspace_bytes < build_rk_ws_bytes(num_kv_heads)) return OSCAR_EWORKSPACE;
    if (!aligned16(q) || !aligned16(rk) || !aligned16(workspace)) return OSCAR_EALIGN;
    cudaError_t e = launch_build_rk(q, n, num_kv_heads, rk, workspace, S(stream));
    return e == cudaSuccess ? OSCAR_OK : cuda_fail(e);
}

size_t oscar_cq_accumulator_bytes(int32_t num_kv_heads) {
    return num_kv_heads > 0 ? cq_acc_bytes(num_kv_heads) : 0;
}

int oscar_cq_reset(void* acc, int32_t num_kv_heads, void* stream) {
    if (!acc || num_kv_heads < 1) return OSCAR_EINVAL;
    if (!aligned16(acc)) return OSCAR_EALIGN;
    cudaError_t e = cudaMemsetAsync(acc, 0, cq_acc_bytes(num_kv_heads), S(stream));
    return e == cudaSuccess ? OSCAR_OK : cuda_fail(e);
}

int oscar_cq_accumulate(const float* q, int64_t n, int32_t num_kv_heads, void* acc, void* stream) {
    if (!acc || num_kv_heads < 1 || n < 0) return OSCAR_EINVAL;
    if (n == 0) return OSCAR_OK;
    if (!q) return OSCAR_EINVAL;
    if (!aligned16(q) || !aligned16(acc)) return OSCAR_EALIGN;
    cudaError_t e = launch_cq_accumulate(q, n, num_kv_heads, acc, S(stream));
    return e == cudaSuccess ? OSCAR_OK : cuda_fail(e);
}

int oscar_cq_finalize(const void* acc, int32_t num_kv_heads, float* rk, void* workspace, size_t workspace_bytes,
                      void* stream) {
    if (!acc || !rk || num_kv_heads < 1) return OSCAR_EINVAL;
    if (!workspace || workspace_bytes < build_rk_ws_bytes(num_kv_heads)) return OSCAR_EWORKSPACE;
    if (!aligned16(acc) || !aligned16(rk) || !aligned16(workspace)) return OSCAR_EALIGN;
    cudaError_t e = launch_cq_finalize(acc, num_kv_heads, rk, workspace, S(stream));
    return e == cudaSuccess ? OSCAR_OK : cuda_fail(e);
}

int oscar_score_weighted_values(const float* q, int64_t n, const float* k, const float* v, int32_t t_keys,
                                int32_t num_kv_heads, float* y, void* stream) {
    if (!q || !k || !v || !y || num_kv_heads < 1 || num_kv_heads > 65535) return OSCAR_EINVAL;
    if (n < 1 || n > INT32_MAX || t_keys < 1 || t_keys > sv_max_keys()) return OSCAR_ERANGE;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(y)) return OSCAR_EALIGN;
    cudaError_t e = launch_score_weighted(q, n, k, v, t_keys, num_kv_heads, y, S(stream));
    return e == cudaSuccess ? OSCAR_OK : cuda_fail(e);
}

// ------------------------------------------------------------------ readback

int oscar_read_int2(const oscar_cache* c, int32_t b, int32_t h, int64_t pos0, int64_t n,
                    uint8_t* k_codes, uint16_t* k_sm, uint8_t* v_codes, uint16_t* v_sm,
                    void* stream) {
    if (!c) return OSCAR_EINVAL;
    if (b < 0 || b >= c->d.batch || h < 0 || h >= c->d.num_kv_heads || n < 0) return OSCAR_ERANGE;
    int64_t l = c->len[b];
    if (n == 0) return OSCAR_OK;
    if (pos0 < kSink || pos0 + n > l - kWindow) return OSCAR_ERANGE;
    const PageFmt f = c->fmt;
    std::vector<uint8_t> blk(f.bytes);
    int64_t cur_page = -1;
    for (int64_t i = 0; i < n; ++i) {
        int64_t pos = pos0 + i;
        int64_t pg = (pos - kSink) / kPage;
        int t = (int)((pos - kSink) % kPage);
        if (pg != cur_page) {
            int32_t phys = c->rows[b][pg];
            const uint8_t* src = c->pool + ((size_t)phys * c->d.num_kv_heads + h) * f.bytes;
            cudaError_t e = cudaMemcpyAsync(blk.data(), src, f.bytes, cudaMemcpyDeviceToHost,
                                            S(stream));
            if (e == cudaSuccess) e = cudaStreamSynchronize(S(stream));
            if (e != cudaSuccess) return cuda_fail(e);
            cur_page = pg;
        }
        if (k_sm) std::memcpy(k_sm + i * (f.k_stride / 2), blk.data() + f.k_sm + t * f.k_stride, f.k_stride);
        if (v_sm) std::memcpy(v_sm + i * (f.v_stride / 2), blk.data() + f.v_sm + t * f.v_stride, f.v_stride);
        // codes: from the page order back to the logical order (channel 4i + j in bits 2j of byte i)
        if (k_codes) {
            uint8_t* dst = k_codes + i * 32;
            std::memset(dst, 0, 32);
            for (int ch = 0; ch < kD; ++ch) {
                int code = (blk[kKCodes + t * 32 + k_code_byte(ch)] >> k_code_shift(ch)) & 3;
                dst[ch / 4] |= (uint8_t)(code << (2 * (ch % 4)));
            }
        }
        if (v_codes) {
            uint8_t* dst = v_codes + i * 32;
            std::memset(dst, 0, 32);
            for (int ch = 0; ch < kD; ++ch) {
                int code = (blk[f.v_codes + v_code_byte(t, ch)] >> v_code_shift(ch)) & 3;
                dst[ch / 4] |= (uint8_t)(code << (2 * (ch % 4)));
            }
        }
    }
    return OSCAR_OK;
}

int oscar_read_bf16(const oscar_cache* c, int32_t b, int32_t h, int64_t pos0, int64_t n,
                    uint16_t* k, uint16_t* v, void* stream) {
    if (!c) return OSCAR_EINVAL;
    if (b < 0 || b >= c->d.batch || h < 0 || h >= c->d.num_kv_heads || n < 0 || pos0 < 0)
        return OSCAR_ERANGE;
    int64_t l = c->len[b];
    for (int64_t pos = pos0; pos < pos0 + n; ++pos) {
        bool sink = pos < std::min<int64_t>(l, kSink);
        bool win = pos >= std::max<int64_t>(kSink, l - kWindow) && pos < l;
        if (!sink && !win) return OSCAR_ERANGE;
    }
    size_t base = ((size_t)b * c->d.num_kv_heads + h) * 2 * kSlots * kD;
    for (int64_t i = 0; i < n; ++i) {
        int slot = bf16_slot(pos0 + i);
        for (int kv = 0; kv < 2; ++kv) {
            uint16_t* dst = kv == 0 ? k : v;
            if (!dst) continue;
            const uint16_t* src = c->bf16 + base + ((size_t)kv * kSlots + slot) * kD;
            cudaError_t e = cudaMemcpyAsync(dst + i * kD, src, kD * sizeof(uint16_t),
                                            cudaMemcpyDeviceToHost, S(stream));
            if (e != cudaSuccess) return cuda_fail(e);
        }
    }
    cudaError_t e = cudaStreamSynchronize(S(stream));
    return e == cudaSuccess ? OSCAR_OK : cuda_fail(e);
}

// ------------------------------------------------------------------ diagnostics

const char* oscar_strerror(int code) {
    switch (code) {
        case OSCAR_OK: return "ok";
        case OSCAR_EINVAL: return "invalid argument";
        case OSCAR_ENOPAGES: return "out of INT2 pages";
        case OSCAR_EWORKSPACE: return "workspace missing or too small";
        case OSCAR_ECUDA: return "CUDA error";
        case OSCAR_EALIGN: return "device pointer not 16-byte aligned";
        case OSCAR_ERANGE: return "index or position out of range";
        case OSCAR_ETIMEOUT: return "a kernel wait timed out";
        case OSCAR_ESCRATCH: return "call needs more than the library's fixed scratch";
        default: return "unknown error";
    }
}

int oscar_last_cuda_error(void) { return g_last_cuda; }

int64_t oscar_launch_count(void) { return g_launches; }

}  // extern "C"

// ------------------------------------------------------------------ fixed-scratch decode (helper)

namespace oscar {

// Fill the parameters of a warp-MMA decode whose scratch is the compact layout
//   rotated queries | one partial per (request, KV head) and per warp | BF16 partials | error word
// inside `scratch` (scratch_bytes long).  Used by oscar_decode_attention_noalloc only.
int noalloc_decode_params(oscar_cache* c, const void* q, int32_t q_dtype, const float* rk, void* out,
                          int32_t out_dtype, void* scratch, size_t scratch_bytes, DecodeParams* pp,
                          cudaStream_t stream) {
    if (!c || !q || !rk || !out || !pp || !scratch) return OSCAR_EINVAL;
    if ((q_dtype != OSCAR_DTYPE_F32 && q_dtype != OSCAR_DTYPE_BF16) ||
        (out_dtype != OSCAR_DTYPE_F32 && out_dtype != OSCAR_DTYPE_BF16))
        return OSCAR_EINVAL;
    if (!aligned16(q) || !aligned16(rk) || !aligned16(out)) return OSCAR_EALIGN;
    DecodeParams& p = *pp;
    std::memset(&p, 0, sizeof(p));
    p.fmt = c->fmt;
    p.batch = c->d.batch;
    p.hkv = c->d.num_kv_heads;
    p.g = c->g;
    p.pps = pick_pps(c);
    p.max_splits = kMaxSplits;
    p.q = q;
    p.q_dtype = q_dtype;
    p.rk = rk;
    p.out = out;
    p.out_dtype = out_dtype;
    p.pool = c->pool;
    p.bf16 = c->bf16;
    p.page_table = c->pt;
    p.max_pps = c->d.max_pages_per_seq;
    p.vmax = c->vmax_dev;
    p.path = OSCAR_PATH_WARP_MMA;
    p.wait_iters = g_wait_iters;
    p.wait_probe = g_wait_probe;
    int64_t pages = 0;
    for (int32_t b = 0; b < c->d.batch; ++b) {
        p.len[b] = (int32_t)c->len[b];
        p.page_off[b] = (int32_t)pages;
        pages += (int64_t)int2_pages(p.len[b]) * c->d.num_kv_heads;
    }
    p.page_off[c->d.batch] = (int32_t)pages;
    if (pages > INT32_MAX / 4) return OSCAR_ERANGE;
    p.total_pages = (int32_t)pages;
    identity_slots(p);
    if (pages > 0) {
        const int rc = mma_unit_count(c->g, pages, &p.n_units);
        if (rc != OSCAR_OK) return rc;
    }
    const size_t per_part = (size_t)c->g * (2 + kD) * sizeof(float);
    const size_t bh = (size_t)c->d.batch * c->d.num_kv_heads;
    const size_t o_err = kNoallocErrOffset;   // fixed, so that oscar_decode_status_noalloc finds it
    const size_t o_qrot = 256;
    const size_t o_mma = o_qrot + (((size_t)c->d.batch * c->d.num_q_heads * kD * sizeof(float) + 255) & ~(size_t)255);
    const size_t o_bf16 = o_mma + (bh + (size_t)p.n_units) * per_part;
    if (o_bf16 + bh * per_part > scratch_bytes) return OSCAR_ESCRATCH;
    uint8_t* ws = (uint8_t*)scratch;
    p.qrot = (float*)(ws + o_qrot);
    p.part_mma = (float*)(ws + o_mma);
    p.part_bf16 = (float*)(ws + o_bf16);
    p.err = (int32_t*)(ws + o_err);
    p.partial = nullptr;   // SIMT partials are not used on the warp-MMA path
    return sync(c, stream);
}

}  // namespace oscar
