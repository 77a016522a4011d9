// zdec.cu -- host runtime behind include/zdec.h: weight upload + repack, the
// paged KV pool (block tables, a page allocator, sequence slots), the
// per-step workspace, the launch sequence of one decode step (replayed as a
// CUDA graph whose kernel edges are programmatic, so each kernel's weight
// prefetch overlaps its predecessor's tail), and the read-backs the parity
// tests use.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "../../include/zdec.h"
#include "zdec_kernels.cuh"

using namespace zdec;

namespace {

thread_local std::string g_global_error;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
// Bytes of a matrix of rows16 row tiles in the grouped layout (padded to whole groups).
size_t tile_bytes(int rows16, int nsb) { return (size_t)n_groups(rows16) * nsb * GROUP_BYTES; }

// Stages a projection consumes per loop step (GemmParams::pair): ZDEC_GEMM_STEP
// = 1 or 2.
int gemm_pair_mode() {
    static const int mode = getenv("ZDEC_GEMM_STEP") ? (atoi(getenv("ZDEC_GEMM_STEP")) == 2 ? 1 : 0) : 1;
    return mode;
}

// K split (cluster size, any 1..16, at least two super-blocks per CTA) for a
// projection whose kernel holds `slots` CTAs on the GPU at once: the split of
// least modelled time, waves x (super-blocks per CTA + 2 for a CTA's fixed
// ramp, reduction and epilogue).  32 row groups of 56 super-blocks split 14
// ways fill 448 of 456 slots in one wave of 4 super-blocks per CTA.
// grid_cap > 0 keeps the grid within that many CTAs (where any split does),
// leaving SM room for the next kernels of the step to become resident early.
template <typename Slots>
int pick_cs(int groups, int nsb, Slots slots_of, int max_cs = 16, int grid_cap = 0) {
    if (groups <= 0) return 1;
    int best = 1;
    double best_t = 1e30;
    for (int cs = 1; cs <= std::min(max_cs, std::max(1, nsb / 2)); cs++) {
        const int slots = slots_of(cs);
        if (slots <= 0) continue;   // the split cannot be launched
        if (grid_cap > 0 && cs > 1 && (long)groups * cs > grid_cap) continue;
        const long waves = ((long)groups * cs + slots - 1) / slots;
        const double t = (double)waves * ((double)nsb / cs + 2.0);
        if (t < best_t - 1e-9) { best_t = t; best = cs; }
    }
    return best;
}
// Batch classes of the split tables: B = 1, <= 4, <= 8, <= 16, <= 32.
int batch_class(int B) { return B == 1 ? 0 : (B <= 4 ? 1 : (B <= 8 ? 2 : (B <= 16 ? 3 : 4))); }
constexpr int CLASS_B[5] = {1, 4, 8, 16, 32};
enum { MAT_QKV, MAT_O, MAT_GU, MAT_DOWN, MAT_LM, N_MAT };
constexpr int MAX_SEGS = 4;   // attention segment slots per row of a step, at most

struct LayerW {
    uint8_t *qkv, *o, *gu, *down;
    float *attn_norm, *ffn_norm;
};

struct Launch {      // one entry of a profiled step
    int kind;
    cudaEvent_t t0, t1;
};

struct AttnPlan {    // attention launch shape for a batch size
    int cs, segs, stages;
};

}  // namespace

struct zdec_ctx {
    zdec_model_desc d{};
    int k_type = 0, v_type = 0, max_B = 0, max_L = 0, Bp_max = 0;
    int qd = 0, kvd = 0, qkv_ld = 0, nsb_h = 0, nsb_f = 0, nsb_q = 0, nrt_vocab = 0;
    int num_sms = 0;
    cudaStream_t stream = nullptr;
    bool own_stream = false;
    // device memory
    uint8_t *wbuf = nullptr;
    size_t wbytes = 0;
    uint8_t *embed = nullptr;
    float *final_norm = nullptr;
    std::vector<LayerW> L;
    // paged KV pool
    KvPool pool{};
    uint8_t *pool_mem = nullptr;
    size_t pool_bytes = 0;
    int max_pages = 0;                 // block-table entries per slot
    std::vector<int> free_pages;       // stack of free page indices
    int32_t *table_host = nullptr;     // pinned mirror of the block tables [max_B][max_pages]
    int32_t *table_dev = nullptr;
    float2 *rope = nullptr;
    void *ws = nullptr;
    size_t ws_bytes = 0;
    float *x = nullptr, *qkv = nullptr, *o = nullptr, *act = nullptr, *logits = nullptr;
    float *amax_v = nullptr;
    int *amax_i = nullptr;
    float *rms_part = nullptr;          // per-group sums of x^2 feeding the next RMSNorm scale
    float *seg_part = nullptr;          // attention partials of rows cut into several segments
    int *seg_ticket = nullptr;
    // GEMM act planes (hi, lo) and sub-block sums: x* for the normed residual,
    // o* for the attention output, a* for the SwiGLU output
    __half *x16 = nullptr, *x16lo = nullptr, *sx = nullptr;
    __half *o16 = nullptr, *o16lo = nullptr, *osx = nullptr;
    __half *a16 = nullptr, *a16lo = nullptr, *asx = nullptr;
    int cs_tab[4][5][N_MAT] = {};   // K split per (projection kernel, batch class, matrix); 0: unset
    int32_t *tok_dev = nullptr, *pos_dev = nullptr, *ids_dev = nullptr, *len_dev = nullptr;
    int32_t *slots_dev = nullptr;      // [max_B] cache slot of each row of a step
    int32_t *ident_dev = nullptr;      // [max_B] 0, 1, 2, ...
    uint32_t *status = nullptr;
    uint4 *qfrag = nullptr;            // [max_B][n_q][32] query fragments (QKV epilogue -> attention)
    int32_t *pinned_io = nullptr;      // [2*max_B] staging of host tokens/positions
    // host state
    std::vector<int> len_host;
    std::vector<int32_t> slots_cur;    // the row -> slot map slots_dev holds (its first slots_n rows)
    int slots_n = 0;
    int gemm_impl = 0, matvec_max_B = 0;
    int b1_impl = 3;                   // projection kernel at B = 1 (ZDEC_B1_IMPL)
    long long wait_limit = 0;  // projection stage-wait bound in clock cycles (0: the kernels' ~2 s)
    std::map<std::tuple<int, const void *, int, int>, cudaGraphExec_t> graphs;   // (B, logits, impl, segments)
    std::string err;
    int last_kernels = 0, last_splits = 0, last_segs = 0;
    // instrumentation of the next/current eager step
    std::vector<Launch> *prof = nullptr;
    float *capture_dev_host = nullptr;   // pinned [L+1][B][H] while a capture is armed
    float *capture_user = nullptr;       // [B][L+1][H]
    bool trace_on = false;               // tracing requested (zdec_set_trace)
    unsigned long long *ktl = nullptr;   // [launches][8] timeline of the last traced step
    unsigned long long *ktl_init = nullptr;   // pinned: its initial values
    size_t ktl_entries = 0;
    std::vector<int> ktl_kinds;          // kernel kind of each launch of the last traced step
};

static zdec_status fail(zdec_ctx *c, zdec_status s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    if (c) c->err = buf;
    else g_global_error = buf;
    return s;
}

#define CK(call)                                                                              \
    do {                                                                                      \
        cudaError_t e_ = (call);                                                              \
        if (e_ != cudaSuccess)                                                                \
            return fail(ctx, ZDEC_ERR_CUDA, "%s failed: %s (%s:%d)", #call,                   \
                        cudaGetErrorString(e_), __FILE__, __LINE__);                          \
    } while (0)

// ---------------------------------------------------------------- create ---
static zdec_status validate_desc(const zdec_model_desc *d) {
    zdec_ctx *ctx = nullptr;
    if (d->n_layers < 1 || d->hidden < 1 || d->n_q_heads < 1 || d->n_kv_heads < 1 || d->vocab < 1 ||
        d->ffn < 1)
        return fail(ctx, ZDEC_ERR_ARG, "model dimensions must be positive");
    if (d->head_dim != HD)
        return fail(ctx, ZDEC_ERR_UNSUPPORTED, "head_dim %d unsupported (kernels implement %d)", d->head_dim, HD);
    if (d->n_q_heads != GROUP * d->n_kv_heads)
        return fail(ctx, ZDEC_ERR_UNSUPPORTED, "n_q_heads must be %d * n_kv_heads", GROUP);
    if (d->hidden % 512 || d->ffn % 512 || (d->n_q_heads * d->head_dim) % 512)
        return fail(ctx, ZDEC_ERR_UNSUPPORTED, "hidden, ffn and n_q_heads*head_dim must be multiples of 512");
    if (!(d->rms_eps >= 0.0f) || !(d->rope_theta > 0.0f))
        return fail(ctx, ZDEC_ERR_ARG, "rms_eps must be >= 0 and rope_theta > 0");
    return ZDEC_OK;
}

static void free_ctx(zdec_ctx *ctx) {
    if (!ctx) return;
    for (auto &kv : ctx->graphs) cudaGraphExecDestroy(kv.second);
    cudaFree(ctx->wbuf);
    cudaFree(ctx->pool_mem);
    cudaFree(ctx->table_dev);
    cudaFreeHost(ctx->table_host);
    cudaFree(ctx->rope);
    cudaFree(ctx->ws);
    cudaFree(ctx->ktl);
    cudaFreeHost(ctx->ktl_init);
    cudaFreeHost(ctx->pinned_io);
    cudaFreeHost(ctx->capture_dev_host);
    if (ctx->own_stream && ctx->stream) cudaStreamDestroy(ctx->stream);
    delete ctx;
}

static zdec_status upload_weights(zdec_ctx *ctx, const zdec_weights *w) {
    const zdec_model_desc &d = ctx->d;
    const int H = d.hidden, F = d.ffn;
    const size_t canon_row_h = (size_t)ctx->nsb_h * CANON_BLOCK;
    const size_t canon_row_f = (size_t)ctx->nsb_f * CANON_BLOCK;
    const size_t canon_row_q = (size_t)ctx->nsb_q * CANON_BLOCK;
    size_t stage_bytes = std::max({(size_t)d.vocab * canon_row_h, (size_t)(ctx->qd + 2 * ctx->kvd) * canon_row_h,
                                   (size_t)2 * F * canon_row_h, (size_t)H * canon_row_f,
                                   (size_t)H * canon_row_q});
    uint8_t *stage = nullptr;
    if (cudaMalloc(&stage, stage_bytes) != cudaSuccess) {
        cudaGetLastError();
        return fail(ctx, ZDEC_ERR_OOM, "cannot allocate %zu bytes of upload staging", stage_bytes);
    }
    auto done = [&](zdec_status s) { cudaFree(stage); return s; };
    auto up = [&](const void *src, size_t off, size_t bytes) -> cudaError_t {
        return cudaMemcpyAsync(stage + off, src, bytes, cudaMemcpyHostToDevice, ctx->stream);
    };
    cudaError_t e;
    // tied embedding / LM head
    if ((e = up(w->embed, 0, (size_t)d.vocab * canon_row_h)) != cudaSuccess ||
        (e = launch_repack(stage, nullptr, 0, d.vocab, ctx->nrt_vocab, ctx->nsb_h, ctx->embed, ctx->stream)) != cudaSuccess ||
        (e = cudaStreamSynchronize(ctx->stream)) != cudaSuccess)
        return done(fail(ctx, ZDEC_ERR_CUDA, "embedding upload: %s", cudaGetErrorString(e)));
    if ((e = cudaMemcpy(ctx->final_norm, w->final_norm, H * sizeof(float), cudaMemcpyHostToDevice)) != cudaSuccess)
        return done(fail(ctx, ZDEC_ERR_CUDA, "final norm upload: %s", cudaGetErrorString(e)));
    for (int l = 0; l < d.n_layers; l++) {
        LayerW &lw = ctx->L[l];
        size_t qb = (size_t)ctx->qd * canon_row_h, kb = (size_t)ctx->kvd * canon_row_h;
        bool ok = (e = up(w->wq[l], 0, qb)) == cudaSuccess && (e = up(w->wk[l], qb, kb)) == cudaSuccess &&
                  (e = up(w->wv[l], qb + kb, kb)) == cudaSuccess &&
                  (e = launch_repack(stage, nullptr, 0, ctx->qd + 2 * ctx->kvd, (ctx->qd + 2 * ctx->kvd) / 16,
                                     ctx->nsb_h, lw.qkv, ctx->stream)) == cudaSuccess &&
                  (e = cudaStreamSynchronize(ctx->stream)) == cudaSuccess;
        ok = ok && (e = up(w->wo[l], 0, (size_t)H * canon_row_q)) == cudaSuccess &&
             (e = launch_repack(stage, nullptr, 0, H, H / 16, ctx->nsb_q, lw.o, ctx->stream)) == cudaSuccess &&
             (e = cudaStreamSynchronize(ctx->stream)) == cudaSuccess;
        size_t gb = (size_t)F * canon_row_h;
        ok = ok && (e = up(w->w_gate[l], 0, gb)) == cudaSuccess && (e = up(w->w_up[l], gb, gb)) == cudaSuccess &&
             (e = launch_repack(stage, stage + gb, 1, F, F / 8, ctx->nsb_h, lw.gu, ctx->stream)) == cudaSuccess &&
             (e = cudaStreamSynchronize(ctx->stream)) == cudaSuccess;
        ok = ok && (e = up(w->w_down[l], 0, (size_t)H * canon_row_f)) == cudaSuccess &&
             (e = launch_repack(stage, nullptr, 0, H, H / 16, ctx->nsb_f, lw.down, ctx->stream)) == cudaSuccess &&
             (e = cudaStreamSynchronize(ctx->stream)) == cudaSuccess;
        ok = ok && (e = cudaMemcpy(lw.attn_norm, w->attn_norm[l], H * sizeof(float), cudaMemcpyHostToDevice)) == cudaSuccess &&
             (e = cudaMemcpy(lw.ffn_norm, w->ffn_norm[l], H * sizeof(float), cudaMemcpyHostToDevice)) == cudaSuccess;
        if (!ok) return done(fail(ctx, ZDEC_ERR_CUDA, "layer %d upload: %s", l, cudaGetErrorString(e)));
    }
    return done(ZDEC_OK);
}

static bool kv_type_ok(int t) { return t == ZDEC_KV_F16 || t == ZDEC_KV_Q8_0 || t == ZDEC_KV_FP8; }

extern "C" zdec_status zdec_create_cache(const zdec_model_desc *desc, const zdec_weights *weights,
                                         const zdec_cache_desc *cache, void *cuda_stream, zdec_ctx **out) {
    zdec_ctx *ctx = nullptr;
    if (!desc || !weights || !cache || !out) return fail(ctx, ZDEC_ERR_ARG, "null argument");
    *out = nullptr;
    zdec_status vs = validate_desc(desc);
    if (vs != ZDEC_OK) return vs;
    if (!kv_type_ok(cache->k_type) || !kv_type_ok(cache->v_type)) return fail(ctx, ZDEC_ERR_ARG, "bad K or V cache type");
    const int max_B = cache->max_B, max_L = cache->max_L;
    if (max_B < 1 || max_B > MAX_B) return fail(ctx, ZDEC_ERR_ARG, "max_B must be in [1, %d]", MAX_B);
    if (max_L < 1) return fail(ctx, ZDEC_ERR_ARG, "max_L must be >= 1");
    if (cache->pool_tokens < 0) return fail(ctx, ZDEC_ERR_ARG, "pool_tokens must be >= 0");
    if (!weights->embed || !weights->final_norm || !weights->attn_norm || !weights->ffn_norm ||
        !weights->wq || !weights->wk || !weights->wv || !weights->wo || !weights->w_gate ||
        !weights->w_up || !weights->w_down)
        return fail(ctx, ZDEC_ERR_ARG, "null weight pointer");

    ctx = new zdec_ctx();
    ctx->d = *desc;
    const zdec_model_desc &d = ctx->d;
    ctx->k_type = cache->k_type;
    ctx->v_type = cache->v_type;
    ctx->max_B = max_B;
    ctx->max_L = max_L;
    ctx->Bp_max = (int)align_up((size_t)max_B, 8);
    ctx->qd = d.n_q_heads * d.head_dim;
    ctx->kvd = d.n_kv_heads * d.head_dim;
    ctx->qkv_ld = ctx->qd + 2 * ctx->kvd;
    ctx->nsb_h = d.hidden / QK;
    ctx->nsb_f = d.ffn / QK;
    ctx->nsb_q = ctx->qd / QK;
    ctx->nrt_vocab = (d.vocab + 15) / 16;
    ctx->L.resize(d.n_layers);
    ctx->len_host.assign(max_B, 0);
    if (const char *e = getenv("ZDEC_MATVEC_MAX_B")) ctx->matvec_max_B = std::max(0, std::min(4, atoi(e)));
    if (const char *e = getenv("ZDEC_B1_IMPL")) ctx->b1_impl = std::max(1, std::min(3, atoi(e)));
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, dev);

    auto bail = [&](zdec_status s) { free_ctx(ctx); return s; };
    if (cuda_stream) ctx->stream = (cudaStream_t)cuda_stream;
    else {
        if (cudaStreamCreateWithFlags(&ctx->stream, cudaStreamNonBlocking) != cudaSuccess)
            return bail(fail(nullptr, ZDEC_ERR_CUDA, "cudaStreamCreate failed"));
        ctx->own_stream = true;
    }
    // ---- weights: one allocation, 256-byte aligned sub-buffers
    const int H = d.hidden, F = d.ffn, NL = d.n_layers;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
    size_t o_embed = take(tile_bytes(ctx->nrt_vocab, ctx->nsb_h));
    size_t o_fn = take(H * sizeof(float));
    std::vector<size_t> oq(NL), oo(NL), og(NL), od(NL), on1(NL), on2(NL);
    for (int l = 0; l < NL; l++) {
        oq[l] = take(tile_bytes((ctx->qd + 2 * ctx->kvd) / 16, ctx->nsb_h));
        oo[l] = take(tile_bytes(H / 16, ctx->nsb_q));
        og[l] = take(tile_bytes(F / 8, ctx->nsb_h));
        od[l] = take(tile_bytes(H / 16, ctx->nsb_f));
        on1[l] = take(H * sizeof(float));
        on2[l] = take(H * sizeof(float));
    }
    ctx->wbytes = off;
    if (cudaMalloc(&ctx->wbuf, ctx->wbytes) != cudaSuccess) {
        cudaGetLastError();
        return bail(fail(nullptr, ZDEC_ERR_OOM, "cannot allocate %zu bytes of weights", ctx->wbytes));
    }
    ctx->embed = ctx->wbuf + o_embed;
    ctx->final_norm = reinterpret_cast<float *>(ctx->wbuf + o_fn);
    for (int l = 0; l < NL; l++)
        ctx->L[l] = {ctx->wbuf + oq[l], ctx->wbuf + oo[l], ctx->wbuf + og[l], ctx->wbuf + od[l],
                     reinterpret_cast<float *>(ctx->wbuf + on1[l]), reinterpret_cast<float *>(ctx->wbuf + on2[l])};

    // ---- paged KV pool: pages of 64 tokens (all layers and kv heads, K and V),
    // one block table per slot
    {
        KvPool &p = ctx->pool;
        p.k_type = ctx->k_type;
        p.v_type = ctx->v_type;
        p.n_layers = NL;
        p.n_kv = d.n_kv_heads;
        p.page_bytes = (size_t)NL * d.n_kv_heads * (kv_region_bytes(p.k_type) + kv_region_bytes(p.v_type));
        ctx->max_pages = (max_L + PAGE_TOKENS - 1) / PAGE_TOKENS;
        const long long want = cache->pool_tokens > 0 ? cache->pool_tokens : (long long)max_B * ctx->max_pages * PAGE_TOKENS;
        const long long pages = (want + PAGE_TOKENS - 1) / PAGE_TOKENS;
        if (pages > (1LL << 30)) return bail(fail(nullptr, ZDEC_ERR_ARG, "pool of %lld pages is too large", pages));
        p.n_pages = (int)pages;
        p.max_pages = ctx->max_pages;
        ctx->pool_bytes = (size_t)p.n_pages * p.page_bytes;
        if (cudaMalloc(&ctx->pool_mem, ctx->pool_bytes) != cudaSuccess) {
            cudaGetLastError();
            return bail(fail(nullptr, ZDEC_ERR_OOM, "cannot allocate the KV pool (%zu bytes: %d pages of %zu)",
                             ctx->pool_bytes, p.n_pages, p.page_bytes));
        }
        p.base = ctx->pool_mem;
        const size_t tb = (size_t)max_B * ctx->max_pages * sizeof(int32_t);
        if (cudaMalloc(&ctx->table_dev, tb) != cudaSuccess || cudaMallocHost(&ctx->table_host, tb) != cudaSuccess) {
            cudaGetLastError();
            return bail(fail(nullptr, ZDEC_ERR_OOM, "cannot allocate the block tables"));
        }
        for (size_t i = 0; i < (size_t)max_B * ctx->max_pages; i++) ctx->table_host[i] = -1;
        if (cudaMemsetAsync(ctx->pool_mem, 0, ctx->pool_bytes, ctx->stream) != cudaSuccess ||
            cudaMemcpyAsync(ctx->table_dev, ctx->table_host, tb, cudaMemcpyHostToDevice, ctx->stream) != cudaSuccess)
            return bail(fail(nullptr, ZDEC_ERR_CUDA, "KV pool initialisation failed"));
        p.table = ctx->table_dev;
        ctx->free_pages.resize(p.n_pages);
        for (int i = 0; i < p.n_pages; i++) ctx->free_pages[i] = p.n_pages - 1 - i;   // page 0 taken first
    }

    // ---- RoPE table [max_L][64] (cos, sin), angles in double
    {
        std::vector<float2> tab((size_t)max_L * (HD / 2));
        std::vector<double> inv(HD / 2);
        for (int i = 0; i < HD / 2; i++) inv[i] = std::pow((double)d.rope_theta, -2.0 * i / HD);
        for (int t = 0; t < max_L; t++)
            for (int i = 0; i < HD / 2; i++) {
                double ang = (double)t * inv[i];
                tab[(size_t)t * (HD / 2) + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
            }
        if (cudaMalloc(&ctx->rope, tab.size() * sizeof(float2)) != cudaSuccess ||
            cudaMemcpy(ctx->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess) {
            cudaGetLastError();
            return bail(fail(nullptr, ZDEC_ERR_OOM, "cannot allocate the RoPE table"));
        }
    }

    // ---- workspace
    {
        const int Bm = max_B, Bp = ctx->Bp_max;
        int lm_grid = n_groups(ctx->nrt_vocab) * 8;   // any cluster split of the LM head
        size_t w = 0;
        auto t = [&](size_t bytes) { size_t o = w; w = align_up(w + bytes, 256); return o; };
        size_t ox = t((size_t)Bm * H * 4), oqkv = t((size_t)Bm * ctx->qkv_ld * 4), oo2 = t((size_t)Bm * ctx->qd * 4);
        size_t oact = t((size_t)Bm * F * 4), olog = t((size_t)Bm * d.vocab * 4);
        size_t oav = t((size_t)lm_grid * MAX_B * 4), oai = t((size_t)lm_grid * MAX_B * 4);
        size_t orms = t((size_t)(n_groups(H / 16) + 1) * MAX_B * 4);
        size_t osp = t((size_t)Bm * MAX_SEGS * d.n_kv_heads * 4 * (HD + 4) * 4);
        size_t ost = t((size_t)MAX_B * d.n_kv_heads * 4);
        auto plane = [&](int K) { return (size_t)(K / QK) * Bp * 256 * 2; };
        auto sums = [&](int K) { return (size_t)(K / QK) * Bp * 16 * 2; };
        size_t ox16 = t(plane(H)), ox16lo = t(plane(H)), osx = t(sums(H));
        size_t oo16 = t(plane(ctx->qd)), oo16lo = t(plane(ctx->qd)), oosx = t(sums(ctx->qd));
        size_t oa16 = t(plane(F)), oa16lo = t(plane(F)), oasx = t(sums(F));
        size_t otok = t(Bm * 4), opos = t(Bm * 4), oids = t(Bm * 4), olen = t(Bm * 4), ostat = t(4);
        size_t oslot = t(Bm * 4), oident = t(Bm * 4);
        size_t oqf = t((size_t)Bm * d.n_q_heads * 32 * 16);
        ctx->ws_bytes = w;
        if (cudaMalloc(&ctx->ws, w) != cudaSuccess) {
            cudaGetLastError();
            return bail(fail(nullptr, ZDEC_ERR_OOM, "cannot allocate %zu bytes of workspace", w));
        }
        uint8_t *b = (uint8_t *)ctx->ws;
        ctx->x = (float *)(b + ox); ctx->qkv = (float *)(b + oqkv); ctx->o = (float *)(b + oo2);
        ctx->act = (float *)(b + oact); ctx->logits = (float *)(b + olog);
        ctx->amax_v = (float *)(b + oav); ctx->amax_i = (int *)(b + oai);
        ctx->rms_part = (float *)(b + orms);
        ctx->seg_part = (float *)(b + osp); ctx->seg_ticket = (int *)(b + ost);
        ctx->x16 = (__half *)(b + ox16); ctx->x16lo = (__half *)(b + ox16lo); ctx->sx = (__half *)(b + osx);
        ctx->o16 = (__half *)(b + oo16); ctx->o16lo = (__half *)(b + oo16lo); ctx->osx = (__half *)(b + oosx);
        ctx->a16 = (__half *)(b + oa16); ctx->a16lo = (__half *)(b + oa16lo); ctx->asx = (__half *)(b + oasx);
        ctx->tok_dev = (int32_t *)(b + otok); ctx->pos_dev = (int32_t *)(b + opos);
        ctx->ids_dev = (int32_t *)(b + oids); ctx->len_dev = (int32_t *)(b + olen);
        ctx->status = (uint32_t *)(b + ostat);
        ctx->slots_dev = (int32_t *)(b + oslot); ctx->ident_dev = (int32_t *)(b + oident);
        ctx->qfrag = (uint4 *)(b + oqf);
        if (cudaMemsetAsync(ctx->ws, 0, w, ctx->stream) != cudaSuccess)
            return bail(fail(nullptr, ZDEC_ERR_CUDA, "workspace memset failed"));
        if (cudaMallocHost(&ctx->pinned_io, 2 * Bm * sizeof(int32_t)) != cudaSuccess)
            return bail(fail(nullptr, ZDEC_ERR_OOM, "cannot allocate pinned staging"));
        std::vector<int32_t> ident(Bm);
        for (int i = 0; i < Bm; i++) ident[i] = i;
        if (cudaStreamSynchronize(ctx->stream) != cudaSuccess ||
            cudaMemcpy(ctx->ident_dev, ident.data(), Bm * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
            cudaMemcpy(ctx->slots_dev, ident.data(), Bm * 4, cudaMemcpyHostToDevice) != cudaSuccess)
            return bail(fail(nullptr, ZDEC_ERR_CUDA, "slot map upload failed"));
        ctx->slots_cur = ident;
        ctx->slots_n = Bm;
    }
    {
        // K splits of every projection for every kernel and batch class, from
        // the occupancy API (ZDEC_CS_MAX: largest split, default 16, a
        // non-portable cluster size)
        const int csmax = getenv("ZDEC_CS_MAX") ? std::max(1, std::min(16, atoi(getenv("ZDEC_CS_MAX")))) : 16;
        // ZDEC_GRID_CAP: projection grids of at most this many CTAs per SM (0: no cap)
        const double gcap = getenv("ZDEC_GRID_CAP") ? atof(getenv("ZDEC_GRID_CAP")) : 0.0;
        const int grid_cap = gcap > 0 ? std::max(1, (int)(gcap * ctx->num_sms)) : 0;
        const int groups[N_MAT] = {n_groups(ctx->qkv_ld / 16), n_groups(H / 16), n_groups(F / 8), n_groups(H / 16),
                                   n_groups(ctx->nrt_vocab)};
        const int nsb[N_MAT] = {ctx->nsb_h, ctx->nsb_q, ctx->nsb_h, ctx->nsb_f, ctx->nsb_h};
        const int epi[N_MAT] = {EPI_STORE, EPI_RESID, EPI_SWIGLU, EPI_RESID, EPI_LMHEAD};
        for (int impl = 1; impl <= 3; impl++)
            for (int c = 0; c < 5; c++) {
                const int Bc = CLASS_B[c];
                if ((impl == 3 && Bc != 1) || (impl == 1 && Bc > 4)) continue;
                for (int m = 0; m < N_MAT; m++)
                    ctx->cs_tab[impl][c][m] = pick_cs(
                        groups[m], nsb[m], [&](int cs) { return gemm_cluster_slots(Bc, impl, epi[m], cs); }, csmax,
                        m == MAT_LM ? 0 : grid_cap);
            }
        cudaGetLastError();
        // ZDEC_SPLITS=q,o,gu,down,lm forces per-matrix splits (0 keeps the model's)
        if (const char *e = getenv("ZDEC_SPLITS")) {
            int f[N_MAT] = {0, 0, 0, 0, 0};
            sscanf(e, "%d,%d,%d,%d,%d", &f[0], &f[1], &f[2], &f[3], &f[4]);
            for (int impl = 1; impl <= 3; impl++)
                for (int c = 0; c < 5; c++)
                    for (int m = 0; m < N_MAT; m++)
                        if (f[m] >= 1 && f[m] <= 16 && ctx->cs_tab[impl][c][m]) ctx->cs_tab[impl][c][m] = f[m];
        }
        if (getenv("ZDEC_PRINT_SPLITS"))   // impl, batch class: splits of qkv, o, gate/up, down, lm head
            for (int impl = 1; impl <= 3; impl++)
                for (int c = 0; c < 5; c++)
                    if (ctx->cs_tab[impl][c][0])
                        fprintf(stderr, "zdec splits impl %d B<=%d: %d %d %d %d %d\n", impl, CLASS_B[c],
                                ctx->cs_tab[impl][c][0], ctx->cs_tab[impl][c][1], ctx->cs_tab[impl][c][2],
                                ctx->cs_tab[impl][c][3], ctx->cs_tab[impl][c][4]);
    }
    if (attention_setup(ctx->k_type, ctx->v_type) != cudaSuccess)
        return bail(fail(nullptr, ZDEC_ERR_CUDA, "attention smem attribute failed"));

    zdec_status us = upload_weights(ctx, weights);
    if (us != ZDEC_OK) {
        g_global_error = ctx->err;
        return bail(us);
    }
    if (cudaStreamSynchronize(ctx->stream) != cudaSuccess)
        return bail(fail(nullptr, ZDEC_ERR_CUDA, "create: %s", cudaGetErrorString(cudaGetLastError())));
    *out = ctx;
    return ZDEC_OK;
}

extern "C" zdec_status zdec_create(const zdec_model_desc *desc, const zdec_weights *weights,
                                   zdec_kv_dtype kv_dtype, int max_B, int max_L, void *cuda_stream,
                                   zdec_ctx **out) {
    zdec_cache_desc c{};
    c.k_type = kv_dtype;
    c.v_type = kv_dtype;
    c.max_B = max_B;
    c.max_L = max_L;
    c.pool_tokens = 0;
    return zdec_create_cache(desc, weights, &c, cuda_stream, out);
}

extern "C" void zdec_destroy(zdec_ctx *ctx) {
    if (!ctx) return;
    cudaStreamSynchronize(ctx->stream);
    free_ctx(ctx);
}

extern "C" const char *zdec_last_error(const zdec_ctx *ctx) { return ctx ? ctx->err.c_str() : g_global_error.c_str(); }
extern "C" const char *zdec_last_global_error(void) { return g_global_error.c_str(); }

// -------------------------------------------------------------- pages ---
// Pages for tokens [t0, t1) of `slot`, taken from the free list where the
// slot has none; the entries set are appended to `fresh`.  On a shortage it
// returns the pages it took and fails with ZDEC_ERR_CAPACITY.
static zdec_status take_pages(zdec_ctx *ctx, int slot, long t0, long t1, std::vector<int> &fresh) {
    if (t1 <= t0) return ZDEC_OK;
    const size_t first = fresh.size();
    for (long pg = t0 / PAGE_TOKENS; pg <= (t1 - 1) / PAGE_TOKENS; pg++) {
        const int e = slot * ctx->max_pages + (int)pg;
        if (ctx->table_host[e] >= 0) continue;
        if (ctx->free_pages.empty()) {
            for (size_t i = first; i < fresh.size(); i++) {
                ctx->free_pages.push_back(ctx->table_host[fresh[i]]);
                ctx->table_host[fresh[i]] = -1;
            }
            fresh.resize(first);
            return fail(ctx, ZDEC_ERR_CAPACITY, "the KV pool has no free page (%d pages of %d tokens)",
                        ctx->pool.n_pages, PAGE_TOKENS);
        }
        ctx->table_host[e] = ctx->free_pages.back();
        ctx->free_pages.pop_back();
        fresh.push_back(e);
    }
    return ZDEC_OK;
}

// Pages listed in `fresh` back to the free list (their entries unset).
static void give_back_pages(zdec_ctx *ctx, std::vector<int> &fresh) {
    for (int e : fresh) {
        ctx->free_pages.push_back(ctx->table_host[e]);
        ctx->table_host[e] = -1;
    }
    fresh.clear();
}

// Block-table entries the host changed, into the device tables (in stream order).
static cudaError_t push_pages(zdec_ctx *ctx, const std::vector<int> &fresh) {
    for (int e : fresh) {
        cudaError_t r = cudaMemcpyAsync(ctx->table_dev + e, ctx->table_host + e, 4, cudaMemcpyHostToDevice, ctx->stream);
        if (r != cudaSuccess) return r;
    }
    return cudaSuccess;
}

// ------------------------------------------------------------- append ---
extern "C" zdec_status zdec_append_kv(zdec_ctx *ctx, int seq, int n_tokens, const void *k_f16,
                                      const void *v_f16, int on_device) {
    if (!ctx) return fail(nullptr, ZDEC_ERR_ARG, "null context");
    if (seq < 0 || seq >= ctx->max_B) return fail(ctx, ZDEC_ERR_ARG, "seq %d out of range", seq);
    if (n_tokens < 0 || (n_tokens > 0 && (!k_f16 || !v_f16))) return fail(ctx, ZDEC_ERR_ARG, "bad tokens/pointers");
    if ((long)ctx->len_host[seq] + n_tokens > ctx->max_L)
        return fail(ctx, ZDEC_ERR_CAPACITY, "sequence %d: %d + %d tokens exceed max_L %d", seq,
                    ctx->len_host[seq], n_tokens, ctx->max_L);
    if (n_tokens == 0) return ZDEC_OK;
    const int t0 = ctx->len_host[seq];
    const zdec_model_desc &d = ctx->d;
    const size_t bytes = (size_t)d.n_layers * n_tokens * d.n_kv_heads * HD * 2;
    void *tmp = nullptr;
    if (!on_device && cudaMalloc(&tmp, 2 * bytes) != cudaSuccess) {
        cudaGetLastError();
        return fail(ctx, ZDEC_ERR_OOM, "cannot stage %zu bytes of KV", 2 * bytes);
    }
    std::vector<int> fresh;
    zdec_status ps = take_pages(ctx, seq, t0, (long)t0 + n_tokens, fresh);
    if (ps != ZDEC_OK) {
        cudaFree(tmp);
        return ps;
    }
    const uint16_t *kd = (const uint16_t *)k_f16, *vd = (const uint16_t *)v_f16;
    cudaError_t e = push_pages(ctx, fresh);
    if (e == cudaSuccess && tmp) {
        e = cudaMemcpyAsync(tmp, k_f16, bytes, cudaMemcpyHostToDevice, ctx->stream);
        if (e == cudaSuccess) e = cudaMemcpyAsync((uint8_t *)tmp + bytes, v_f16, bytes, cudaMemcpyHostToDevice, ctx->stream);
        kd = (const uint16_t *)tmp;
        vd = (const uint16_t *)((uint8_t *)tmp + bytes);
    }
    if (e == cudaSuccess) e = launch_kv_append(ctx->pool, seq, t0, n_tokens, kd, vd, ctx->status, ctx->stream);
    int32_t newlen = t0 + n_tokens;
    if (e == cudaSuccess) e = cudaMemcpyAsync(ctx->len_dev + seq, &newlen, 4, cudaMemcpyHostToDevice, ctx->stream);
    cudaError_t e2 = cudaStreamSynchronize(ctx->stream);   // the host length source is read asynchronously
    cudaFree(tmp);
    if (e == cudaSuccess) e = e2;
    if (e != cudaSuccess) return fail(ctx, ZDEC_ERR_CUDA, "append_kv: %s", cudaGetErrorString(e));
    ctx->len_host[seq] = newlen;
    return ZDEC_OK;
}

extern "C" zdec_status zdec_reset_seq(zdec_ctx *ctx, int seq) {
    if (!ctx) return fail(nullptr, ZDEC_ERR_ARG, "null context");
    if (seq < 0 || seq >= ctx->max_B) return fail(ctx, ZDEC_ERR_ARG, "seq %d out of range", seq);
    CK(cudaStreamSynchronize(ctx->stream));   // no step in flight still reads the slot's pages
    std::vector<int> freed;
    for (int pg = 0; pg < ctx->max_pages; pg++) {
        const int e = seq * ctx->max_pages + pg;
        if (ctx->table_host[e] >= 0) {
            ctx->free_pages.push_back(ctx->table_host[e]);
            ctx->table_host[e] = -1;
            freed.push_back(e);
        }
    }
    int32_t zero = 0;
    CK(push_pages(ctx, freed));
    CK(cudaMemcpyAsync(ctx->len_dev + seq, &zero, 4, cudaMemcpyHostToDevice, ctx->stream));
    CK(cudaStreamSynchronize(ctx->stream));
    ctx->len_host[seq] = 0;
    return ZDEC_OK;
}

extern "C" zdec_status zdec_seq_len(const zdec_ctx *ctx, int seq, int *len) {
    if (!ctx || !len) return fail(nullptr, ZDEC_ERR_ARG, "null argument");
    if (seq < 0 || seq >= ctx->max_B) return ZDEC_ERR_ARG;
    *len = ctx->len_host[seq];
    return ZDEC_OK;
}

// --------------------------------------------------------------- step ---
// Attention ring depth.  A deeper ring pays off only where the attention
// dominates the step; elsewhere its shared memory keeps the neighbouring
// projections' CTAs (which prefetch their weights) off the SMs.
static int attn_stages(const zdec_ctx *ctx, int B) {
    static const int env = getenv("ZDEC_ATT_STAGES") ? atoi(getenv("ZDEC_ATT_STAGES")) : 0;
    const int lim = attention_stage_limit(ctx->k_type, ctx->v_type);
    if (env >= 2) return std::min(env, lim);
    (void)B;
    return std::min(lim, 3);   // measured: 3 beats 2 at B = 1 and 8, fp16 and one-byte types; 4 adds nothing
}
// Segment slots per row for a step whose rows hold these many tokens: one
// when the rows are about even (a cut row pays a cross-segment merge, ~3 us
// at B = 1 measured), up to MAX_SEGS when the longest row is that many times
// the mean, so that its clusters take about a mean row's work each; the ratio
// is rounded to nearest (measured at B = 8: lengths 800..30,000, ratio 3.26,
// 3 / 4 slots 4.11 / 3.82 ms with fp16 but 3.71 / 3.89 ms with Q8_0; lengths
// 6,000 + 7 x 2,000, ratio 2.4, 2 / 3 slots 2.76 / 2.85 ms).
static int attn_segments(const zdec_ctx *ctx, int B) {
    static const int f_seg = getenv("ZDEC_ATT_SEGS") ? atoi(getenv("ZDEC_ATT_SEGS")) : 0;
    if (f_seg >= 1) return std::min(f_seg, MAX_SEGS);
    long sum = 0, mx = 0;
    for (int b = 0; b < B; b++) {
        const long n = ctx->len_host[ctx->slots_cur[b]] + 1;
        sum += n;
        mx = std::max(mx, n);
    }
    const double ratio = sum > 0 ? (double)mx * B / (double)sum : 1.0;
    return std::max(1, std::min(MAX_SEGS, (int)(ratio + 0.5)));
}
// Attention launch shape for a batch of B rows cut into `segs` segment slots
// per row: the cluster size cs (ranks per segment) of least modelled time,
// waves x (chunks per CTA + 1 for the query load and the cluster merge), for
// a nominal 64 chunks per row, the waves from the occupancy API's co-resident
// clusters (which must each fit one GPC).  ZDEC_ATT_CS forces one.
static AttnPlan attn_plan(const zdec_ctx *ctx, int B, int segs) {
    static const int f_cs = getenv("ZDEC_ATT_CS") ? atoi(getenv("ZDEC_ATT_CS")) : 0;
    AttnPlan best{1, segs, attn_stages(ctx, B)};
    double best_t = 1e30;
    for (int m = segs; m <= segs; m++) {
        for (int cs = 1; cs <= 16; cs++) {
            if (f_cs >= 1 && f_cs <= 16 && cs != f_cs) continue;
            const int maxc = attention_max_clusters(ctx->k_type, ctx->v_type, best.stages, cs, ctx->d.n_kv_heads);
            if (maxc <= 0) continue;
            const int clusters = B * ctx->d.n_kv_heads * m;
            const double t = (double)((clusters + maxc - 1) / maxc) * (64.0 / (m * cs) + 1.0);
            if (t < best_t - 1e-9) { best_t = t; best.cs = cs; best.segs = m; }
        }
    }
    if (getenv("ZDEC_PRINT_SPLITS"))
        fprintf(stderr, "zdec attention B=%d: %d stages, cluster %d, %d segment slot(s) per row\n", B, best.stages,
                best.cs, best.segs);
    return best;
}

static int pick_impl(const zdec_ctx *ctx, int B) {
    if (B > 4) return 2;
    if (ctx->gemm_impl == 1) return 1;
    if (ctx->gemm_impl == 2) return 2;
    if (ctx->gemm_impl == 3) return B == 1 ? 3 : 2;
    if (B == 1) return ctx->b1_impl;
    return B <= ctx->matvec_max_B ? 1 : 2;
}

// Enqueue the whole step for rows 0..B-1 (row b uses cache slot slots_dev[b]),
// the attention cut into `segs` segment slots per row.  logits_out may be null.
static cudaError_t enqueue_step(zdec_ctx *ctx, int B, int segs, float *logits_out, bool pdl) {
    const zdec_model_desc &d = ctx->d;
    const int H = d.hidden, F = d.ffn;
    const int impl = pick_impl(ctx, B);
    cudaStream_t s = ctx->stream;
    int nk = 0;
    cudaError_t e;
    auto mark = [&](int kind, bool begin) {
        if (!ctx->prof) return;
        if (begin) {
            Launch L{kind, nullptr, nullptr};
            cudaEventCreate(&L.t0);
            cudaEventCreate(&L.t1);
            cudaEventRecord(L.t0, s);
            ctx->prof->push_back(L);
        } else {
            cudaEventRecord(ctx->prof->back().t1, s);
        }
    };
    auto capture_x = [&](int slot) -> cudaError_t {
        if (!ctx->capture_dev_host) return cudaSuccess;
        return cudaMemcpyAsync(ctx->capture_dev_host + (size_t)slot * B * H, ctx->x, (size_t)B * H * 4,
                               cudaMemcpyDeviceToHost, s);
    };
    // launch timeline (tracing): slot nk of ctx->ktl for launch nk
    unsigned long long *tlb = ctx->trace_on ? ctx->ktl : nullptr, *tlk = nullptr;
    if (tlb) {
        ctx->ktl_kinds.clear();
        if ((e = cudaMemcpyAsync(tlb, ctx->ktl_init, ctx->ktl_entries * 8, cudaMemcpyHostToDevice, s)) != cudaSuccess)
            return e;
    }
#define STEP(kind, call)                        \
    do {                                        \
        tlk = tlb ? tlb + 8 * nk : nullptr;     \
        if (tlb) ctx->ktl_kinds.push_back(kind); \
        mark(kind, true);                       \
        if ((e = (call)) != cudaSuccess)        \
            return e;                           \
        mark(kind, false);                      \
        nk++;                                   \
    } while (0)

    const int Bp0 = ctx->Bp_max;
    const int bc = batch_class(B);   // split-table row
    auto split = [&](int m) { const int c = ctx->cs_tab[impl][bc][m]; return c > 0 ? c : 1; };
    STEP(ZDEC_KERNEL_EMBED, launch_embed(ctx->embed, ctx->nsb_h, d.vocab, ctx->tok_dev, ctx->pos_dev, ctx->slots_dev,
                                         ctx->len_dev, ctx->status, B, ctx->x, H, ctx->L[0].attn_norm,
                                         ctx->x16, ctx->x16lo, ctx->sx, Bp0, ctx->rms_part, pdl, s, tlk));
    if ((e = capture_x(0)) != cudaSuccess) return e;
    const int Bp = ctx->Bp_max;   // row pitch of every act plane
    GemmParams gp{};
    gp.B = B;
    gp.Bp = Bp;
    gp.out_Bp = Bp;
    gp.status = ctx->status;
    gp.wait_limit = ctx->wait_limit;
    gp.pair = gemm_pair_mode();
    // Every projection takes its activation as fp16 hi + lo planes (~22 bits):
    // the new K/V rows are rounded and quantized, and over dozens of layers a
    // single fp16 operand would drift past the parity tolerance.
    auto operand = [&](__half *hi, __half *lo, __half *sums) { gp.x16 = hi; gp.x16lo = lo; gp.sx = sums; };
    auto matrix = [&](const uint8_t *W, int N, int nrt, int nsb, int cs) {
        gp.W = W; gp.N = N; gp.nrt = nrt; gp.nsb = nsb; gp.cs = cs;
    };
    const AttnPlan plan = attn_plan(ctx, B, segs);
    AttnParams ap{};
    ap.kv = ctx->pool;
    ap.nq = d.n_q_heads;
    ap.positions = ctx->pos_dev;
    ap.slots = ctx->slots_dev;
    ap.qkv = ctx->qkv;
    ap.qkv_ld = ctx->qkv_ld;
    ap.rope = ctx->rope;
    ap.append = 1;
    ap.cs = plan.cs;
    ap.seg_min = 2;
    ap.stages = plan.stages;
    ap.o = nullptr;   // the O projection reads the operand planes only
    ap.o16 = ctx->o16;
    ap.o16lo = ctx->o16lo;
    ap.osx = ctx->osx;
    ap.oBp = Bp;
    ap.B = B;
    ap.max_L = ctx->max_L;
    ap.status = ctx->status;
    ap.q_frag = ctx->qfrag;   // written by the QKV projection's epilogue
    ap.seg_part = ctx->seg_part;
    ap.seg_ticket = ctx->seg_ticket;
    const int nz = B * plan.segs;
    // RMSNorm never runs as its own kernel: the producer of the residual (the
    // embedding gather, the O and down projections) writes gain*x as the next
    // projection's operand plus per-group sums of x^2, and the consumer scales
    // its outputs by r = 1/sqrt(mean x^2 + eps).
    const int resid_groups = n_groups(H / 16);
    auto normed_input = [&](int nparts) {
        operand(ctx->x16, ctx->x16lo, ctx->sx);
        gp.rms_part = ctx->rms_part; gp.rms_nparts = nparts; gp.rms_K = H; gp.rms_eps = d.rms_eps;
    };
    auto plain_input = [&](__half *hi, __half *lo, __half *sums) {
        operand(hi, lo, sums);
        gp.rms_part = nullptr;
    };
    for (int l = 0; l < d.n_layers; l++) {
        const LayerW &lw = ctx->L[l];
        normed_input(l == 0 ? 1 : resid_groups);
        matrix(lw.qkv, ctx->qkv_ld, ctx->qkv_ld / 16, ctx->nsb_h, split(MAT_QKV));
        gp.out = ctx->qkv; gp.ldo = ctx->qkv_ld;
        gp.q_frag = ctx->qfrag; gp.q_pos = ctx->pos_dev; gp.q_rope = ctx->rope; gp.q_heads = d.n_q_heads;
        STEP(ZDEC_KERNEL_GEMM_QKV, (gp.tl = tlk, launch_gemm(gp, EPI_STORE, impl, pdl, s)));
        gp.q_frag = nullptr;
        ap.layer = l;
        STEP(ZDEC_KERNEL_ATTENTION, (ap.tl = tlk, launch_attention(ap, nz, pdl, s)));
        plain_input(ctx->o16, ctx->o16lo, ctx->osx);   // written by the attention merge
        matrix(lw.o, H, H / 16, ctx->nsb_q, split(MAT_O));
        gp.out = ctx->x; gp.ldo = H;
        gp.next_gain = lw.ffn_norm; gp.part_out = ctx->rms_part;
        gp.out16 = ctx->x16; gp.out16lo = ctx->x16lo; gp.out_sx = ctx->sx;
        STEP(ZDEC_KERNEL_GEMM_O, (gp.tl = tlk, launch_gemm(gp, EPI_RESID, impl, pdl, s)));
        normed_input(resid_groups);
        matrix(lw.gu, F, F / 8, ctx->nsb_h, split(MAT_GU));
        gp.out = nullptr; gp.ldo = F;
        gp.out16 = ctx->a16; gp.out16lo = ctx->a16lo; gp.out_sx = ctx->asx;
        STEP(ZDEC_KERNEL_GEMM_GATEUP, (gp.tl = tlk, launch_gemm(gp, EPI_SWIGLU, impl, pdl, s)));
        plain_input(ctx->a16, ctx->a16lo, ctx->asx);   // written by the gate/up epilogue
        matrix(lw.down, H, H / 16, ctx->nsb_f, split(MAT_DOWN));
        gp.out = ctx->x; gp.ldo = H;
        gp.next_gain = l + 1 < d.n_layers ? ctx->L[l + 1].attn_norm : ctx->final_norm;
        gp.part_out = ctx->rms_part;
        gp.out16 = ctx->x16; gp.out16lo = ctx->x16lo; gp.out_sx = ctx->sx;
        STEP(ZDEC_KERNEL_GEMM_DOWN, (gp.tl = tlk, launch_gemm(gp, EPI_RESID, impl, pdl, s)));
        if ((e = capture_x(l + 1)) != cudaSuccess) return e;
    }
    normed_input(resid_groups);
    matrix(ctx->embed, d.vocab, ctx->nrt_vocab, ctx->nsb_h, split(MAT_LM));
    gp.out = logits_out; gp.ldo = d.vocab;
    gp.amax_val = ctx->amax_v; gp.amax_idx = ctx->amax_i;
    STEP(ZDEC_KERNEL_GEMM_LMHEAD, (gp.tl = tlk, launch_gemm(gp, EPI_LMHEAD, impl, pdl, s)));
    STEP(ZDEC_KERNEL_ARGMAX, launch_argmax_final(ctx->amax_v, ctx->amax_i, n_groups(ctx->nrt_vocab), B, ctx->ids_dev,
                                                 ctx->pos_dev, ctx->slots_dev, ctx->len_dev, ctx->status, pdl, s, tlk));
#undef STEP
    ctx->last_kernels = nk;
    ctx->last_splits = plan.cs;
    ctx->last_segs = plan.segs;
    return cudaSuccess;
}

// Host checks of a step: row count, distinct in-range slots, room in every
// slot, and a page for every new token (taken here; `fresh` lists the block
// table entries set).  On failure nothing has changed.
static zdec_status check_step_args(zdec_ctx *ctx, int B, const int32_t *slots, const int32_t *tokens,
                                   const int32_t *positions, int32_t *ids, std::vector<int> &fresh) {
    if (!ctx) return fail(nullptr, ZDEC_ERR_ARG, "null context");
    if (B < 1 || B > ctx->max_B) return fail(ctx, ZDEC_ERR_ARG, "B=%d outside [1, %d]", B, ctx->max_B);
    if (!tokens || !positions || !ids) return fail(ctx, ZDEC_ERR_ARG, "null tokens/positions/ids");
    std::vector<char> used(ctx->max_B, 0);
    for (int b = 0; b < B; b++) {
        const int s = slots ? slots[b] : b;
        if (s < 0 || s >= ctx->max_B) return fail(ctx, ZDEC_ERR_ARG, "slots[%d] = %d outside [0, %d)", b, s, ctx->max_B);
        if (used[s]) return fail(ctx, ZDEC_ERR_ARG, "slot %d appears twice in one step", s);
        used[s] = 1;
    }
    for (int b = 0; b < B; b++) {
        const int s = slots ? slots[b] : b;
        if (ctx->len_host[s] + 1 > ctx->max_L)
            return fail(ctx, ZDEC_ERR_CAPACITY, "slot %d is full (%d tokens)", s, ctx->max_L);
    }
    for (int b = 0; b < B; b++) {
        const int s = slots ? slots[b] : b;
        zdec_status ps = take_pages(ctx, s, ctx->len_host[s], (long)ctx->len_host[s] + 1, fresh);
        if (ps != ZDEC_OK) {   // the pages earlier rows took go back
            give_back_pages(ctx, fresh);
            return ps;
        }
    }
    return ZDEC_OK;
}

// The row -> slot map of this step into slots_dev (only when it changed; it
// then waits for the steps in flight, which read the old map).
static zdec_status set_slots(zdec_ctx *ctx, int B, const int32_t *slots) {
    bool same = B <= ctx->slots_n;
    for (int b = 0; same && b < B; b++) same = ctx->slots_cur[b] == (slots ? slots[b] : b);
    if (same) return ZDEC_OK;
    CK(cudaStreamSynchronize(ctx->stream));
    for (int b = 0; b < B; b++) ctx->slots_cur[b] = slots ? slots[b] : b;
    CK(cudaMemcpy(ctx->slots_dev, ctx->slots_cur.data(), B * 4, cudaMemcpyHostToDevice));
    ctx->slots_n = B;
    return ZDEC_OK;
}

// Host-I/O input checks (before anything is enqueued): every row's position
// is its slot's length, every token is in the vocabulary.
static zdec_status check_host_inputs(zdec_ctx *ctx, int B, const int32_t *slots, const int32_t *tokens,
                                     const int32_t *positions) {
    for (int b = 0; b < B; b++) {
        const int s = slots ? slots[b] : b;
        if (positions[b] != ctx->len_host[s])
            return fail(ctx, ZDEC_ERR_POSITION, "positions[%d] = %d but slot %d holds %d tokens", b, positions[b], s,
                        ctx->len_host[s]);
        if (tokens[b] < 0 || tokens[b] >= ctx->d.vocab)
            return fail(ctx, ZDEC_ERR_ARG, "tokens[%d] = %d outside the vocabulary", b, tokens[b]);
    }
    return ZDEC_OK;
}

// Stage inputs: host inputs go through pinned memory.
static zdec_status stage_inputs(zdec_ctx *ctx, int B, const int32_t *tokens, const int32_t *positions, bool host) {
    if (host) {
        CK(cudaStreamSynchronize(ctx->stream));   // the pinned staging may still be in flight
        memcpy(ctx->pinned_io, tokens, B * 4);
        memcpy(ctx->pinned_io + ctx->max_B, positions, B * 4);
        CK(cudaMemcpyAsync(ctx->tok_dev, ctx->pinned_io, B * 4, cudaMemcpyHostToDevice, ctx->stream));
        CK(cudaMemcpyAsync(ctx->pos_dev, ctx->pinned_io + ctx->max_B, B * 4, cudaMemcpyHostToDevice, ctx->stream));
    } else {
        CK(cudaMemcpyAsync(ctx->tok_dev, tokens, B * 4, cudaMemcpyDeviceToDevice, ctx->stream));
        CK(cudaMemcpyAsync(ctx->pos_dev, positions, B * 4, cudaMemcpyDeviceToDevice, ctx->stream));
    }
    return ZDEC_OK;
}

// Everything before the kernels of a step: host checks, pages, the slot map
// and the inputs.  When it fails the step has changed nothing.
static zdec_status prepare_step(zdec_ctx *ctx, int B, const int32_t *slots, const int32_t *tokens,
                                const int32_t *positions, int32_t *ids, bool host) {
    std::vector<int> fresh;
    zdec_status st = check_step_args(ctx, B, slots, tokens, positions, ids, fresh);
    if (st != ZDEC_OK) return st;
    if (host) st = check_host_inputs(ctx, B, slots, tokens, positions);
    if (st == ZDEC_OK) st = set_slots(ctx, B, slots);
    if (st == ZDEC_OK) st = stage_inputs(ctx, B, tokens, positions, host);
    if (st != ZDEC_OK) {
        give_back_pages(ctx, fresh);
        return st;
    }
    cudaError_t e = push_pages(ctx, fresh);
    if (e != cudaSuccess) return fail(ctx, ZDEC_ERR_CUDA, "block table update: %s", cudaGetErrorString(e));
    return ZDEC_OK;
}

static zdec_status run_step(zdec_ctx *ctx, int B, const int32_t *slots, const int32_t *tokens,
                            const int32_t *positions, float *logits, int32_t *ids, int flags) {
    const bool host = flags & ZDEC_STEP_HOST_IO;
    zdec_status st = prepare_step(ctx, B, slots, tokens, positions, ids, host);
    if (st != ZDEC_OK) return st;
    const bool eager = (flags & ZDEC_STEP_EAGER) || ctx->capture_dev_host || ctx->trace_on;
    float *lg = host ? (logits ? ctx->logits : nullptr) : logits;
    const int impl = pick_impl(ctx, B);
    const int segs = attn_segments(ctx, B);
    if (eager) {
        CK(enqueue_step(ctx, B, segs, lg, true));
    } else {
        auto key = std::make_tuple(B, (const void *)lg, impl, segs);
        auto it = ctx->graphs.find(key);
        if (it == ctx->graphs.end()) {
            cudaGraph_t graph;
            CK(cudaStreamBeginCapture(ctx->stream, cudaStreamCaptureModeThreadLocal));
            cudaError_t e = enqueue_step(ctx, B, segs, lg, true);
            cudaError_t e2 = cudaStreamEndCapture(ctx->stream, &graph);
            if (e != cudaSuccess || e2 != cudaSuccess) {
                if (e2 == cudaSuccess) cudaGraphDestroy(graph);
                return fail(ctx, ZDEC_ERR_CUDA, "step capture: %s", cudaGetErrorString(e != cudaSuccess ? e : e2));
            }
            cudaGraphExec_t exec;
            cudaError_t e3 = cudaGraphInstantiate(&exec, graph, 0);
            cudaGraphDestroy(graph);
            if (e3 != cudaSuccess) return fail(ctx, ZDEC_ERR_CUDA, "graph instantiate: %s", cudaGetErrorString(e3));
            it = ctx->graphs.emplace(key, exec).first;
        }
        CK(cudaGraphLaunch(it->second, ctx->stream));
    }
    if (host) {
        if (logits)
            CK(cudaMemcpyAsync(logits, ctx->logits, (size_t)B * ctx->d.vocab * 4, cudaMemcpyDeviceToHost, ctx->stream));
        CK(cudaMemcpyAsync(ids, ctx->ids_dev, B * 4, cudaMemcpyDeviceToHost, ctx->stream));
    } else {
        CK(cudaMemcpyAsync(ids, ctx->ids_dev, B * 4, cudaMemcpyDeviceToDevice, ctx->stream));
    }
    for (int b = 0; b < B; b++) ctx->len_host[ctx->slots_cur[b]]++;
    if (ctx->capture_dev_host) {   // armed hidden-state capture: wait and reorder
        cudaError_t e = cudaStreamSynchronize(ctx->stream);
        const int H = ctx->d.hidden, NL1 = ctx->d.n_layers + 1;
        if (e == cudaSuccess)
            for (int b = 0; b < B; b++)
                for (int l = 0; l < NL1; l++)
                    memcpy(ctx->capture_user + ((size_t)b * NL1 + l) * H,
                           ctx->capture_dev_host + ((size_t)l * B + b) * H, (size_t)H * sizeof(float));
        cudaFreeHost(ctx->capture_dev_host);
        ctx->capture_dev_host = nullptr;
        ctx->capture_user = nullptr;
        if (e != cudaSuccess) return fail(ctx, ZDEC_ERR_CUDA, "captured step: %s", cudaGetErrorString(e));
    }
    if (host) return zdec_sync(ctx);
    return ZDEC_OK;
}

extern "C" zdec_status zdec_decode_step(zdec_ctx *ctx, int B, const int32_t *tokens,
                                        const int32_t *positions, float *logits, int32_t *ids, int flags) {
    return run_step(ctx, B, nullptr, tokens, positions, logits, ids, flags);
}

extern "C" zdec_status zdec_decode_step_slots(zdec_ctx *ctx, int B, const int32_t *slots, const int32_t *tokens,
                                              const int32_t *positions, float *logits, int32_t *ids, int flags) {
    if (ctx && !slots) return fail(ctx, ZDEC_ERR_ARG, "null slots");
    return run_step(ctx, B, slots, tokens, positions, logits, ids, flags);
}

extern "C" zdec_status zdec_sync(zdec_ctx *ctx) {
    if (!ctx) return fail(nullptr, ZDEC_ERR_ARG, "null context");
    CK(cudaStreamSynchronize(ctx->stream));
    uint32_t st = 0;
    CK(cudaMemcpy(&st, ctx->status, 4, cudaMemcpyDeviceToHost));
    if (st) {
        uint32_t zero = 0;
        CK(cudaMemcpy(ctx->status, &zero, 4, cudaMemcpyHostToDevice));
        // the flagged steps advanced no device length, while the host mirror
        // counted every step it enqueued: take the device's lengths back
        std::vector<int32_t> len(ctx->max_B);
        CK(cudaMemcpy(len.data(), ctx->len_dev, ctx->max_B * sizeof(int32_t), cudaMemcpyDeviceToHost));
        for (int b = 0; b < ctx->max_B; b++) ctx->len_host[b] = len[b];
        if (st & STATUS_TIMEOUT) return fail(ctx, ZDEC_ERR_TIMEOUT, "a bounded device wait gave up");
        return fail(ctx, ZDEC_ERR_DEVICE, "device check failed (status 0x%x:%s%s%s)", st,
                    (st & STATUS_POSITION) ? " position != cached length" : "",
                    (st & STATUS_TOKEN) ? " token outside the vocabulary" : "",
                    (st & STATUS_PAGE) ? " cached token without a KV page" : "");
    }
    return ZDEC_OK;
}

extern "C" zdec_status zdec_debug_set_wait_limit(zdec_ctx *ctx, long long cycles) {
    if (!ctx) return fail(nullptr, ZDEC_ERR_ARG, "null context");
    if (cycles < -1) return fail(ctx, ZDEC_ERR_ARG, "cycles must be >= -1");
    CK(cudaStreamSynchronize(ctx->stream));
    for (auto &kv : ctx->graphs) cudaGraphExecDestroy(kv.second);   // they captured the old bound
    ctx->graphs.clear();
    ctx->wait_limit = cycles;
    return ZDEC_OK;
}

extern "C" zdec_status zdec_set_gemm_impl(zdec_ctx *ctx, int impl) {
    if (!ctx) return fail(nullptr, ZDEC_ERR_ARG, "null context");
    if (impl < 0 || impl > 3) return fail(ctx, ZDEC_ERR_ARG, "impl must be 0, 1, 2 or 3");
    ctx->gemm_impl = impl;
    return ZDEC_OK;
}

extern "C" zdec_status zdec_get_info(const zdec_ctx *ctx, zdec_info *info) {
    if (!ctx || !info) return fail(nullptr, ZDEC_ERR_ARG, "null argument");
    info->weight_bytes = ctx->wbytes;
    info->arena_bytes = ctx->pool_bytes;
    info->workspace_bytes = ctx->ws_bytes;
    info->kv_bytes_per_token = ctx->pool.page_bytes / PAGE_TOKENS;
    info->kernels_per_step = ctx->last_kernels;
    info->attn_splits = ctx->last_splits;
    info->matvec_max_B = ctx->matvec_max_B;
    info->attn_segments = ctx->last_segs;
    info->k_type = ctx->k_type;
    info->v_type = ctx->v_type;
    info->page_tokens = PAGE_TOKENS;
    info->pool_pages = ctx->pool.n_pages;
    info->free_pages = (int)ctx->free_pages.size();
    return ZDEC_OK;
}

extern "C" zdec_status zdec_set_trace(zdec_ctx *ctx, int on) {
    if (!ctx) return fail(nullptr, ZDEC_ERR_ARG, "null context");
    CK(cudaStreamSynchronize(ctx->stream));
    if (!on) {
        cudaFree(ctx->ktl);
        cudaFreeHost(ctx->ktl_init);
        ctx->ktl = nullptr;
        ctx->ktl_init = nullptr;
        ctx->ktl_entries = 0;
        ctx->trace_on = false;
        return ZDEC_OK;
    }
    if (ctx->trace_on) return ZDEC_OK;
    // [launches][8] = (first start, first past the wait, last end, kind, milestones)
    const size_t nk = (size_t)(3 + 5 * ctx->d.n_layers) * 8;
    if (cudaMalloc(&ctx->ktl, nk * 8) != cudaSuccess || cudaMallocHost(&ctx->ktl_init, nk * 8) != cudaSuccess) {
        cudaGetLastError();
        return fail(ctx, ZDEC_ERR_OOM, "cannot allocate the launch timeline");
    }
    for (size_t i = 0; i < nk; i++) ctx->ktl_init[i] = (i % 8 < 2) ? ~0ULL : 0ULL;
    ctx->ktl_entries = nk;
    ctx->trace_on = true;
    return ZDEC_OK;
}

extern "C" zdec_status zdec_debug_step_trace(zdec_ctx *ctx, uint64_t *out_host, size_t cap, size_t *n) {
    if (!ctx || !n) return fail(nullptr, ZDEC_ERR_ARG, "null argument");
    *n = ctx->trace_on ? ctx->ktl_entries : 0;
    if (!ctx->trace_on || !out_host || *n == 0) return ZDEC_OK;   // size query
    if (cap < *n) return fail(ctx, ZDEC_ERR_ARG, "trace needs %zu entries", *n);
    CK(cudaStreamSynchronize(ctx->stream));
    CK(cudaMemcpy(out_host, ctx->ktl, *n * 8, cudaMemcpyDeviceToHost));
    for (size_t i = 0; i < *n / 8; i++) out_host[8 * i + 3] = i < ctx->ktl_kinds.size() ? ctx->ktl_kinds[i] : 0;
    return ZDEC_OK;
}

extern "C" zdec_status zdec_profile_step(zdec_ctx *ctx, int B, const int32_t *tokens_dev,
                                         const int32_t *positions_dev, float *logits_dev, int32_t *ids_dev,
                                         int *kind, float *ms, int cap, int *n) {
    if (ctx && (!n || (cap > 0 && (!kind || !ms)))) return fail(ctx, ZDEC_ERR_ARG, "null output");
    zdec_status st = prepare_step(ctx, B, nullptr, tokens_dev, positions_dev, ids_dev, false);
    if (st != ZDEC_OK) return st;
    std::vector<Launch> launches;
    ctx->prof = &launches;
    cudaError_t e = enqueue_step(ctx, B, attn_segments(ctx, B), logits_dev, false);
    ctx->prof = nullptr;
    if (e == cudaSuccess) e = cudaMemcpyAsync(ids_dev, ctx->ids_dev, B * 4, cudaMemcpyDeviceToDevice, ctx->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
    for (size_t i = 0; i < launches.size(); i++) {
        float t = 0.0f;
        if (e == cudaSuccess) cudaEventElapsedTime(&t, launches[i].t0, launches[i].t1);
        if ((int)i < cap) { kind[i] = launches[i].kind; ms[i] = t; }
        cudaEventDestroy(launches[i].t0);
        cudaEventDestroy(launches[i].t1);
    }
    *n = (int)launches.size();
    if (e != cudaSuccess) return fail(ctx, ZDEC_ERR_CUDA, "profile step: %s", cudaGetErrorString(e));
    for (int b = 0; b < B; b++) ctx->len_host[ctx->slots_cur[b]]++;
    return zdec_sync(ctx);
}

// -------------------------------------------------------------- debug ---
static zdec_status tensor_info(zdec_ctx *ctx, int which, int layer, const uint8_t *&tiles, int &row_map,
                               int &row_off, int &rows, int &nsb) {
    const zdec_model_desc &d = ctx->d;
    if (which != ZDEC_T_EMBED && (layer < 0 || layer >= d.n_layers)) return fail(ctx, ZDEC_ERR_ARG, "bad layer");
    row_map = 0;
    row_off = 0;
    switch (which) {
        case ZDEC_T_EMBED: tiles = ctx->embed; rows = d.vocab; nsb = ctx->nsb_h; break;
        case ZDEC_T_WQ: tiles = ctx->L[layer].qkv; rows = ctx->qd; nsb = ctx->nsb_h; break;
        case ZDEC_T_WK: tiles = ctx->L[layer].qkv; row_off = ctx->qd; rows = ctx->kvd; nsb = ctx->nsb_h; break;
        case ZDEC_T_WV: tiles = ctx->L[layer].qkv; row_off = ctx->qd + ctx->kvd; rows = ctx->kvd; nsb = ctx->nsb_h; break;
        case ZDEC_T_WO: tiles = ctx->L[layer].o; rows = d.hidden; nsb = ctx->nsb_q; break;
        case ZDEC_T_GATE: tiles = ctx->L[layer].gu; row_map = 1; rows = d.ffn; nsb = ctx->nsb_h; break;
        case ZDEC_T_UP: tiles = ctx->L[layer].gu; row_map = 2; rows = d.ffn; nsb = ctx->nsb_h; break;
        case ZDEC_T_DOWN: tiles = ctx->L[layer].down; rows = d.hidden; nsb = ctx->nsb_f; break;
        default: return fail(ctx, ZDEC_ERR_ARG, "bad tensor id %d", which);
    }
    return ZDEC_OK;
}

template <typename P, typename F>
static zdec_status debug_rows(zdec_ctx *ctx, int which, int layer, int row0, int nrows, void *out, P per_row,
                              F launch) {
    if (!ctx || !out) return fail(ctx, ZDEC_ERR_ARG, "null argument");
    const uint8_t *tiles;
    int row_map, row_off, rows, nsb;
    zdec_status st = tensor_info(ctx, which, layer, tiles, row_map, row_off, rows, nsb);
    if (st != ZDEC_OK) return st;
    if (row0 < 0 || nrows < 0 || row0 + nrows > rows) return fail(ctx, ZDEC_ERR_ARG, "rows out of range");
    if (nrows == 0) return ZDEC_OK;
    void *dbuf = nullptr;
    size_t bytes = (size_t)nrows * per_row(nsb);
    if (cudaMalloc(&dbuf, bytes) != cudaSuccess) { cudaGetLastError(); return fail(ctx, ZDEC_ERR_OOM, "debug buffer"); }
    cudaError_t e = launch(tiles, row_map, nsb, row_off + row0, nrows, dbuf);
    if (e == cudaSuccess) e = cudaMemcpyAsync(out, dbuf, bytes, cudaMemcpyDeviceToHost, ctx->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
    cudaFree(dbuf);
    if (e != cudaSuccess) return fail(ctx, ZDEC_ERR_CUDA, "debug read: %s", cudaGetErrorString(e));
    return ZDEC_OK;
}

extern "C" zdec_status zdec_debug_export_q4k(zdec_ctx *ctx, int which, int layer, int row0, int nrows, void *out_host) {
    return debug_rows(ctx, which, layer, row0, nrows, out_host,
                      [](int nsb) { return (size_t)nsb * CANON_BLOCK; },
                      [&](const uint8_t *t, int rm, int nsb, int r0, int nr, void *dst) {
                          return launch_export_canonical(t, rm, nsb, r0, nr, (uint8_t *)dst, ctx->stream);
                      });
}

extern "C" zdec_status zdec_debug_dequant(zdec_ctx *ctx, int which, int layer, int row0, int nrows, float *out_host) {
    return debug_rows(ctx, which, layer, row0, nrows, out_host,
                      [](int nsb) { return (size_t)nsb * QK * sizeof(float); },
                      [&](const uint8_t *t, int rm, int nsb, int r0, int nr, void *dst) {
                          return launch_dequant_rows(t, rm, nsb, r0, nr, (float *)dst, ctx->stream);
                      });
}

extern "C" zdec_status zdec_debug_read_kv(zdec_ctx *ctx, int seq, int layer, int t0, int n, void *k, void *v,
                                          void *ks, void *vs) {
    if (!ctx || !k || !v) return fail(ctx, ZDEC_ERR_ARG, "null argument");
    if ((ctx->k_type == ZDEC_KV_Q8_0 && !ks) || (ctx->v_type == ZDEC_KV_Q8_0 && !vs))
        return fail(ctx, ZDEC_ERR_ARG, "a Q8_0 tensor's read needs its scale buffer");
    if (seq < 0 || seq >= ctx->max_B || layer < 0 || layer >= ctx->d.n_layers || t0 < 0 || n < 0 ||
        t0 + n > ctx->max_L)
        return fail(ctx, ZDEC_ERR_ARG, "range out of bounds");
    if (n == 0) return ZDEC_OK;
    const int nkv = ctx->d.n_kv_heads;
    const size_t kb = (size_t)n * nkv * HD * (ctx->k_type == ZDEC_KV_F16 ? 2 : 1);
    const size_t vb = (size_t)n * nkv * HD * (ctx->v_type == ZDEC_KV_F16 ? 2 : 1);
    const size_t sb = (size_t)n * nkv * 4 * 2;
    uint8_t *buf = nullptr;
    if (cudaMalloc(&buf, kb + vb + 2 * sb + 16) != cudaSuccess) { cudaGetLastError(); return fail(ctx, ZDEC_ERR_OOM, "debug buffer"); }
    uint16_t *dks = (uint16_t *)(buf + kb + vb), *dvs = (uint16_t *)(buf + kb + vb + sb);
    cudaError_t e = launch_kv_read(ctx->pool, seq, layer, t0, n, buf, buf + kb, dks, dvs, ctx->stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(k, buf, kb, cudaMemcpyDeviceToHost, ctx->stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(v, buf + kb, vb, cudaMemcpyDeviceToHost, ctx->stream);
    if (e == cudaSuccess && ctx->k_type == ZDEC_KV_Q8_0) e = cudaMemcpyAsync(ks, dks, sb, cudaMemcpyDeviceToHost, ctx->stream);
    if (e == cudaSuccess && ctx->v_type == ZDEC_KV_Q8_0) e = cudaMemcpyAsync(vs, dvs, sb, cudaMemcpyDeviceToHost, ctx->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
    cudaFree(buf);
    if (e != cudaSuccess) return fail(ctx, ZDEC_ERR_CUDA, "kv read: %s", cudaGetErrorString(e));
    return ZDEC_OK;
}

extern "C" zdec_status zdec_debug_block_table(zdec_ctx *ctx, int seq, int32_t *pages_host, int cap, int *n) {
    if (!ctx || !n) return fail(ctx, ZDEC_ERR_ARG, "null argument");
    if (seq < 0 || seq >= ctx->max_B) return fail(ctx, ZDEC_ERR_ARG, "seq %d out of range", seq);
    *n = ctx->max_pages;
    if (!pages_host) return ZDEC_OK;
    if (cap < ctx->max_pages) return fail(ctx, ZDEC_ERR_ARG, "the table needs %d entries", ctx->max_pages);
    CK(cudaStreamSynchronize(ctx->stream));
    CK(cudaMemcpy(pages_host, ctx->table_dev + (size_t)seq * ctx->max_pages, ctx->max_pages * 4, cudaMemcpyDeviceToHost));
    return ZDEC_OK;
}

extern "C" zdec_status zdec_debug_capture_hidden(zdec_ctx *ctx, float *out_host) {
    if (!ctx || !out_host) return fail(ctx, ZDEC_ERR_ARG, "null argument");
    if (!ctx->capture_dev_host) {
        size_t bytes = (size_t)(ctx->d.n_layers + 1) * ctx->max_B * ctx->d.hidden * sizeof(float);
        if (cudaMallocHost(&ctx->capture_dev_host, bytes) != cudaSuccess) {
            cudaGetLastError();
            return fail(ctx, ZDEC_ERR_OOM, "cannot allocate %zu pinned bytes for the capture", bytes);
        }
    }
    ctx->capture_user = out_host;
    return ZDEC_OK;
}

extern "C" zdec_status zdec_debug_attention(zdec_ctx *ctx, int layer, int B, const float *q_host,
                                            const int32_t *positions_host, float *o_host) {
    if (!ctx || !q_host || !positions_host || !o_host) return fail(ctx, ZDEC_ERR_ARG, "null argument");
    if (B < 1 || B > ctx->max_B || layer < 0 || layer >= ctx->d.n_layers) return fail(ctx, ZDEC_ERR_ARG, "bad B/layer");
    for (int b = 0; b < B; b++)
        if (positions_host[b] < 0 || positions_host[b] >= ctx->len_host[b])
            return fail(ctx, ZDEC_ERR_ARG, "position %d of row %d is not a cached token", positions_host[b], b);
    const int qd = ctx->qd;
    CK(cudaMemcpy2DAsync(ctx->qkv, ctx->qkv_ld * 4, q_host, qd * 4, qd * 4, B, cudaMemcpyHostToDevice, ctx->stream));
    CK(cudaMemcpyAsync(ctx->pos_dev, positions_host, B * 4, cudaMemcpyHostToDevice, ctx->stream));
    std::vector<int32_t> saved(ctx->slots_cur);   // the segment choice reads rows 0..B-1 as slots 0..B-1
    for (int b = 0; b < B; b++) ctx->slots_cur[b] = b;
    const AttnPlan plan = attn_plan(ctx, B, attn_segments(ctx, B));
    ctx->slots_cur = saved;
    AttnParams ap{};
    ap.kv = ctx->pool;
    ap.layer = layer;
    ap.nq = ctx->d.n_q_heads;
    ap.positions = ctx->pos_dev;
    ap.slots = ctx->ident_dev;   // row b reads slot b
    ap.qkv = ctx->qkv;
    ap.qkv_ld = ctx->qkv_ld;
    ap.rope = ctx->rope;
    ap.append = 0;
    ap.cs = plan.cs;
    ap.seg_min = 2;
    ap.stages = plan.stages;
    ap.o = ctx->o;
    ap.o16 = ctx->o16;
    ap.o16lo = ctx->o16lo;
    ap.osx = ctx->osx;
    ap.oBp = ctx->Bp_max;
    ap.B = B;
    ap.max_L = ctx->max_L;
    ap.status = ctx->status;
    ap.seg_part = ctx->seg_part;
    ap.seg_ticket = ctx->seg_ticket;
    CK(launch_attention(ap, B * plan.segs, false, ctx->stream));
    CK(cudaMemcpyAsync(o_host, ctx->o, (size_t)B * qd * 4, cudaMemcpyDeviceToHost, ctx->stream));
    CK(cudaStreamSynchronize(ctx->stream));
    return ZDEC_OK;
}

// ---------------------------------------------------------- stateless ---
extern "C" size_t zdec_q4k_repacked_bytes(int N, int K) {
    if (N <= 0 || K <= 0 || N % 16 || K % QK) return 0;
    return tile_bytes(N / 16, K / QK);
}

extern "C" zdec_status zdec_q4k_repack(const void *canonical_dev, int N, int K, void *repacked_dev, void *stream) {
    zdec_ctx *ctx = nullptr;
    if (!canonical_dev || !repacked_dev) return fail(ctx, ZDEC_ERR_ARG, "null pointer");
    if (N <= 0 || N % 16 || K <= 0 || K % 512) return fail(ctx, ZDEC_ERR_UNSUPPORTED, "N must be a multiple of 16 and K of 512");
    CK(launch_repack((const uint8_t *)canonical_dev, nullptr, 0, N, N / 16, K / QK, (uint8_t *)repacked_dev,
                     (cudaStream_t)stream));
    return ZDEC_OK;
}

extern "C" size_t zdec_q4k_gemm_workspace_bytes(int K, int B) {
    if (K <= 0 || K % QK || B < 1 || B > MAX_B) return 0;
    const size_t plane = align_up((size_t)(K / QK) * B * 256 * 2, 256);
    return 2 * plane + (size_t)(K / QK) * B * 16 * 2 + 256;
}

// Argument checks shared by the two stateless projection entry points.
static zdec_status check_q4k_gemm(const void *repacked_dev, int N, int K, const float *x_dev, int B,
                                  const float *y_dev, int impl) {
    zdec_ctx *ctx = nullptr;
    if (!repacked_dev || !x_dev || !y_dev) return fail(ctx, ZDEC_ERR_ARG, "null pointer");
    if (N <= 0 || N % 16 || K <= 0 || K % 512) return fail(ctx, ZDEC_ERR_UNSUPPORTED, "N must be a multiple of 16 and K of 512");
    if (B < 1 || B > MAX_B) return fail(ctx, ZDEC_ERR_ARG, "B must be in [1, %d]", MAX_B);
    if (impl < 1 || impl > 3) return fail(ctx, ZDEC_ERR_ARG, "impl must be 1, 2 or 3");
    if (impl == 1 && B > 4) return fail(ctx, ZDEC_ERR_UNSUPPORTED, "the matvec handles B <= 4");
    if (impl == 3 && B != 1) return fail(ctx, ZDEC_ERR_UNSUPPORTED, "impl 3 handles B = 1");
    if ((uintptr_t)x_dev % 16) return fail(ctx, ZDEC_ERR_ARG, "x_dev must be 16-byte aligned");
    return ZDEC_OK;
}

// The projection itself on checked arguments, with its scratch (hi plane, lo
// plane, sub-block sums; zdec_q4k_gemm_workspace_bytes(K, B) bytes) at `scratch`.
static zdec_status run_q4k_gemm(const void *repacked_dev, int N, int K, const float *x_dev, int B, float *y_dev,
                                int impl, void *scratch, cudaStream_t s) {
    zdec_ctx *ctx = nullptr;
    const size_t plane = align_up((size_t)(K / QK) * B * 256 * 2, 256);
    __half *hi = (__half *)scratch;
    __half *lo = (__half *)((uint8_t *)scratch + plane);
    __half *sums = (__half *)((uint8_t *)scratch + 2 * plane);
    CK(launch_prep(x_dev, K, K, nullptr, 0.0f, B, B, hi, lo, sums, false, s));
    GemmParams gp{};
    gp.W = (const uint8_t *)repacked_dev;
    gp.N = N;
    gp.nrt = N / 16;
    gp.nsb = K / QK;
    gp.x16 = hi;
    gp.x16lo = lo;
    gp.sx = sums;
    gp.B = B;
    gp.Bp = B;
    gp.out = y_dev;
    gp.ldo = N;
    gp.cs = pick_cs(n_groups(N / 16), K / QK, [&](int cs) { return gemm_cluster_slots(B, impl, EPI_STORE, cs); });
    gp.pair = gemm_pair_mode();
    CK(launch_gemm(gp, EPI_STORE, impl, false, s));
    return ZDEC_OK;
}

extern "C" zdec_status zdec_q4k_gemm(const void *repacked_dev, int N, int K, const float *x_dev, int B, float *y_dev,
                                     int impl, void *workspace_dev, size_t workspace_bytes, void *stream) {
    zdec_ctx *ctx = nullptr;
    zdec_status st = check_q4k_gemm(repacked_dev, N, K, x_dev, B, y_dev, impl);
    if (st != ZDEC_OK) return st;
    if (!workspace_dev) return fail(ctx, ZDEC_ERR_ARG, "null workspace");
    if (workspace_bytes < zdec_q4k_gemm_workspace_bytes(K, B)) return fail(ctx, ZDEC_ERR_ARG, "workspace too small");
    if ((uintptr_t)workspace_dev % 16) return fail(ctx, ZDEC_ERR_ARG, "pointers must be 16-byte aligned");
    return run_q4k_gemm(repacked_dev, N, K, x_dev, B, y_dev, impl, workspace_dev, (cudaStream_t)stream);
}

// ------------------------------------------------- allocation-free GEMM ---
// The stateless projection for callers that cannot hand over device memory:
// a plain C host with no device allocator of its own, or a caller inside a
// section that must not call cudaMalloc/cudaFree (cudaFree waits for the
// whole device, stalling every other stream).  The activation planes that
// zdec_q4k_gemm keeps in the caller's workspace live here in one file-scope
// device array, sized for K*B <= ZDEC_Q4K_GEMM_STATIC_MAX_KB, with the same
// layout (hi plane, lo plane, sub-block sums).  Nothing in it has to start at
// zero: each call's prep kernel writes every byte its GEMM then reads.
namespace {
constexpr size_t kStaticPlaneBytes = (size_t)ZDEC_Q4K_GEMM_STATIC_MAX_KB * 2;   // a multiple of 256
constexpr size_t kStaticScratchBytes =
    2 * kStaticPlaneBytes + (size_t)ZDEC_Q4K_GEMM_STATIC_MAX_KB / QK * 16 * 2 + 256;
constexpr int kStaticMaxDevices = 64;
std::mutex g_static_mu;
void *g_static_addr[kStaticMaxDevices];   // device address of the array, looked up once per device
}  // namespace

static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

extern "C" zdec_status zdec_q4k_gemm_static(const void *repacked_dev, int N, int K, const float *x_dev, int B,
                                            float *y_dev, int impl, void *stream) {
    zdec_ctx *ctx = nullptr;
    zdec_status st = check_q4k_gemm(repacked_dev, N, K, x_dev, B, y_dev, impl);
    if (st != ZDEC_OK) return st;
    if ((long long)K * B > ZDEC_Q4K_GEMM_STATIC_MAX_KB)
        return fail(ctx, ZDEC_ERR_ARG,
                    "K*B = %lld exceeds the static scratch of zdec_q4k_gemm_static (K*B <= %d); "
                    "use zdec_q4k_gemm with a caller workspace",
                    (long long)K * B, ZDEC_Q4K_GEMM_STATIC_MAX_KB);
    int dev = 0;
    CK(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kStaticMaxDevices) return fail(ctx, ZDEC_ERR_UNSUPPORTED, "device ordinal %d too large", dev);
    void *base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_static_mu);
        if (!g_static_addr[dev]) CK(cudaGetSymbolAddress(&g_static_addr[dev], g_static_scratch));
        base = g_static_addr[dev];
    }
    return run_q4k_gemm(repacked_dev, N, K, x_dev, B, y_dev, impl, base, (cudaStream_t)stream);
}
