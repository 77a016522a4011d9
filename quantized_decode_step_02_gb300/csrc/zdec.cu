// zdec.cu -- host runtime behind include/zdec.h: weight upload + repack, the
// KV arena, the per-step workspace, the launch sequence of one decode step
// (replayed as a CUDA graph whose kernel edges are programmatic, so each
// kernel's weight prefetch overlaps its predecessor's tail), and the
// read-backs the parity tests use.
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

// Projection pipeline mode (GemmParams::pipe): 0 (stage pairs) unless
// ZDEC_GEMM_PIPE=1; pairs measured faster, their two independent stages
// giving each warp more instruction-level parallelism.
int gemm_pipe_mode() {
    static const int mode = getenv("ZDEC_GEMM_PIPE") ? (atoi(getenv("ZDEC_GEMM_PIPE")) ? 1 : 0) : 0;
    return mode;
}

// K split (cluster size, any 1..16, at least two super-blocks per CTA) for a
// projection whose kernel holds `slots` CTAs on the GPU at once: the split of
// least modelled time, waves x (super-blocks per CTA + 2 for a CTA's fixed
// ramp, reduction and epilogue).  32 row groups of 56 super-blocks split 14
// ways fill 448 of 456 slots in one wave of 4 super-blocks per CTA.
template <typename Slots>
int pick_cs(int groups, int nsb, Slots slots_of, int max_cs = 16) {
    if (groups <= 0) return 1;
    int best = 1;
    double best_t = 1e30;
    for (int cs = 1; cs <= std::min(max_cs, std::max(1, nsb / 2)); cs++) {
        const int slots = slots_of(cs);
        if (slots <= 0) continue;   // the split cannot be launched
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

struct LayerW {
    uint8_t *qkv, *o, *gu, *down;
    float *attn_norm, *ffn_norm;
};

struct Launch {      // one entry of a profiled step
    int kind;
    cudaEvent_t t0, t1;
};

}  // namespace

struct zdec_ctx {
    zdec_model_desc d{};
    int kv_dtype = 0, max_B = 0, max_L = 0, Lp = 0, Bp_max = 0;
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
    KvArena arena{};
    size_t arena_bytes = 0;
    std::vector<void *> arena_allocs;
    float2 *rope = nullptr;
    void *ws = nullptr;
    size_t ws_bytes = 0;
    float *x = nullptr, *qkv = nullptr, *o = nullptr, *act = nullptr, *logits = nullptr;
    float *part = nullptr, *amax_v = nullptr;
    int *amax_i = nullptr, *tickets = nullptr;
    float *rms_part = nullptr;          // per-group sums of x^2 feeding the next RMSNorm scale
    // GEMM act planes (hi, lo) and sub-block sums: x* for the normed residual,
    // o* for the attention output, a* for the SwiGLU output
    __half *x16 = nullptr, *x16lo = nullptr, *sx = nullptr;
    __half *o16 = nullptr, *o16lo = nullptr, *osx = nullptr;
    __half *a16 = nullptr, *a16lo = nullptr, *asx = nullptr;
    int cs_tab[4][5][N_MAT] = {};   // K split per (projection kernel, batch class, matrix); 0: unset
    int32_t *tok_dev = nullptr, *pos_dev = nullptr, *ids_dev = nullptr, *len_dev = nullptr;
    uint32_t *status = nullptr;
    uint4 *qfrag = nullptr;            // [max_B][n_q][32] query fragments (QKV epilogue -> attention)
    int32_t *pinned_io = nullptr;      // [2*max_B] staging of host tokens/positions
    // host state
    std::vector<int> len_host;
    int gemm_impl = 0, matvec_max_B = 0;
    int b1_impl = 3;                   // projection kernel at B = 1 (ZDEC_B1_IMPL)
    size_t prefetch_cap = 0;   // bytes of the next matrix a GEMM warms in L2 (0: off; ZDEC_L2_PREFETCH_MB)
    long long wait_limit = 0;  // projection stage-wait bound in clock cycles (0: the kernels' ~2 s)
    std::map<std::tuple<int, const void *, int>, cudaGraphExec_t> graphs;
    std::string err;
    int last_kernels = 0, last_splits = 0;
    // instrumentation of the next/current eager step
    std::vector<Launch> *prof = nullptr;
    float *capture_dev_host = nullptr;   // pinned [L+1][B][H] while a capture is armed
    float *capture_user = nullptr;       // [B][L+1][H]
    // persistent step kernel (step.cu)
    int engine = ZDEC_ENGINE_AUTO, last_engine = ZDEC_ENGINE_KERNELS;
    int step_grid = 0;                   // CTAs (0: the persistent kernel is unavailable)
    int step_slots[2] = {0, 0};          // ring slots for B <= 4 and B <= 8
    void *step_buf = nullptr;            // its buffers (one allocation)
    StepLayerW *d_layers = nullptr;
    float *s_q = nullptr, *s_gpart = nullptr, *s_apart = nullptr, *s_rms_ffn = nullptr, *s_capture = nullptr;
    __half *g16 = nullptr, *g16lo = nullptr, *gsx = nullptr;
    int *s_cnt = nullptr, *s_ok = nullptr, *s_abort = nullptr;
    int s_ncnt = 0;
    bool persistent_eager = false;       // its CUDA graph capture failed: launch it directly
    int step_pf_items = 0;               // L2 prefetch distance (items per CTA; ZDEC_STEP_PF_ITEMS)
    int step_att_min = 8;                // attention units per CTA at least (ZDEC_STEP_ATT_MIN)
    unsigned long long *trace = nullptr; // phase timeline of the last persistent step, or null
    size_t trace_entries = 0;
    bool trace_on = false;               // tracing requested (zdec_set_trace)
    unsigned long long *ktl = nullptr;   // kernel engine: [launches][4] timeline of the last step
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
    for (void *p : ctx->arena_allocs) cudaFree(p);
    cudaFree(ctx->rope);
    cudaFree(ctx->ws);
    cudaFree(ctx->step_buf);
    cudaFree(ctx->trace);
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

// Ring slots and CTAs of the persistent step kernel, and its buffers.  The
// kernel runs two CTAs per SM when they fit (one otherwise); it is left
// unavailable (step_grid = 0) when the device cannot launch it cooperatively,
// or when the attention output width differs from the hidden size.
static zdec_status step_configure(zdec_ctx *ctx) {
    const zdec_model_desc &d = ctx->d;
    int dev = 0, coop = 0, smem_sm = 0, reserved = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (getenv("ZDEC_NO_PERSISTENT") || !coop || ctx->qd != d.hidden || ctx->num_sms < 1) return ZDEC_OK;
    if (const char *e = getenv("ZDEC_STEP_PF_ITEMS")) ctx->step_pf_items = std::max(0, atoi(e));
    if (const char *e = getenv("ZDEC_STEP_ATT_MIN")) ctx->step_att_min = std::max(1, atoi(e));
    int per_sm = 2;
    for (int v = 0; v < 2; v++) {
        const int B = v ? STEP_MAX_B : 4;
        const size_t static_smem = 11 * 1024;   // the kernel's own __shared__ state
        int slots = (int)(((size_t)smem_sm / 2 - reserved - static_smem) / (step_slot_bytes(B) + 16));
        // the attention's warp pairs need a slot count divisible by their number (<= 4)
        slots = std::max(2, std::min(8, slots));
        if (slots == 5) slots = 4;
        if (slots == 7) slots = 6;
        int fit = 0;
        while (true) {
            if (step_setup(B, ctx->kv_dtype, slots, &fit) != cudaSuccess) {
                cudaGetLastError();
                return ZDEC_OK;
            }
            if (fit >= 2 || slots <= 2) break;
            slots = slots == 6 ? 4 : slots - 1;
        }
        if (fit < 1) return ZDEC_OK;
        per_sm = std::min(per_sm, fit);
        ctx->step_slots[v] = slots;
    }
    const int grid = per_sm * ctx->num_sms;
    const int H = d.hidden, NL = d.n_layers, Bm = std::min(ctx->max_B, STEP_MAX_B);
    ctx->s_ncnt = step_counter_count(NL, H, d.ffn, d.vocab, d.n_q_heads, d.n_kv_heads);
    size_t w = 0;
    auto t = [&](size_t bytes) { size_t o = w; w = align_up(w + bytes, 256); return o; };
    auto plane = [&](int K) { return (size_t)(K / QK) * Bm * 256 * 2; };
    const size_t o_layers = t(sizeof(StepLayerW) * NL);
    const size_t o_q = t((size_t)Bm * ctx->qd * 4);
    const size_t o_gp = t(step_gpart_floats(H, d.ffn, d.vocab, d.n_q_heads, d.n_kv_heads, Bm, grid) * 4);
    const size_t o_ap = t(step_apart_floats(d.n_kv_heads, Bm, grid) * 4);
    const size_t o_rf = t((size_t)(H / 128) * MAX_B * 4);
    const size_t o_cap = t((size_t)(NL + 1) * Bm * H * 4);
    const size_t o_g = t(plane(H)), o_glo = t(plane(H)), o_gsx = t((size_t)(H / QK) * Bm * 16 * 2);
    const size_t o_cnt = t((size_t)ctx->s_ncnt * 4), o_ok = t(4), o_ab = t(4);
    if (cudaMalloc(&ctx->step_buf, w) != cudaSuccess) {
        cudaGetLastError();
        return fail(nullptr, ZDEC_ERR_OOM, "cannot allocate %zu bytes for the step kernel", w);
    }
    uint8_t *b = (uint8_t *)ctx->step_buf;
    ctx->d_layers = (StepLayerW *)(b + o_layers);
    ctx->s_q = (float *)(b + o_q);
    ctx->s_gpart = (float *)(b + o_gp);
    ctx->s_apart = (float *)(b + o_ap);
    ctx->s_rms_ffn = (float *)(b + o_rf);
    ctx->s_capture = (float *)(b + o_cap);
    ctx->g16 = (__half *)(b + o_g);
    ctx->g16lo = (__half *)(b + o_glo);
    ctx->gsx = (__half *)(b + o_gsx);
    ctx->s_cnt = (int *)(b + o_cnt);
    ctx->s_ok = (int *)(b + o_ok);
    ctx->s_abort = (int *)(b + o_ab);
    std::vector<StepLayerW> lw(NL);
    for (int l = 0; l < NL; l++)
        lw[l] = {ctx->L[l].qkv, ctx->L[l].o, ctx->L[l].gu, ctx->L[l].down, ctx->L[l].attn_norm, ctx->L[l].ffn_norm};
    if (cudaMemsetAsync(ctx->step_buf, 0, w, ctx->stream) != cudaSuccess ||
        cudaMemcpyAsync(ctx->d_layers, lw.data(), sizeof(StepLayerW) * NL, cudaMemcpyHostToDevice, ctx->stream) !=
            cudaSuccess ||
        cudaStreamSynchronize(ctx->stream) != cudaSuccess)
        return fail(nullptr, ZDEC_ERR_CUDA, "step kernel buffers: %s", cudaGetErrorString(cudaGetLastError()));
    ctx->step_grid = grid;
    return ZDEC_OK;
}

extern "C" zdec_status zdec_create(const zdec_model_desc *desc, const zdec_weights *weights,
                                   zdec_kv_dtype kv_dtype, int max_B, int max_L, void *cuda_stream,
                                   zdec_ctx **out) {
    zdec_ctx *ctx = nullptr;
    if (!desc || !weights || !out) return fail(ctx, ZDEC_ERR_ARG, "null argument");
    *out = nullptr;
    zdec_status vs = validate_desc(desc);
    if (vs != ZDEC_OK) return vs;
    if (kv_dtype != ZDEC_KV_F16 && kv_dtype != ZDEC_KV_Q8_0) return fail(ctx, ZDEC_ERR_ARG, "bad kv_dtype");
    if (max_B < 1 || max_B > MAX_B) return fail(ctx, ZDEC_ERR_ARG, "max_B must be in [1, %d]", MAX_B);
    if (max_L < 1) return fail(ctx, ZDEC_ERR_ARG, "max_L must be >= 1");
    if (!weights->embed || !weights->final_norm || !weights->attn_norm || !weights->ffn_norm ||
        !weights->wq || !weights->wk || !weights->wv || !weights->wo || !weights->w_gate ||
        !weights->w_up || !weights->w_down)
        return fail(ctx, ZDEC_ERR_ARG, "null weight pointer");

    ctx = new zdec_ctx();
    ctx->d = *desc;
    const zdec_model_desc &d = ctx->d;
    ctx->kv_dtype = kv_dtype;
    ctx->max_B = max_B;
    ctx->max_L = max_L;
    ctx->Lp = (int)align_up((size_t)max_L, ATT_CHUNK);
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
    if (const char *e = getenv("ZDEC_L2_PREFETCH_MB")) ctx->prefetch_cap = (size_t)std::max(0, atoi(e)) << 20;
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

    // ---- KV arena
    KvArena &a = ctx->arena;
    a.kv_dtype = kv_dtype;
    a.n_layers = NL;
    a.n_kv = d.n_kv_heads;
    a.Lp = ctx->Lp;
    size_t planes = (size_t)max_B * NL * d.n_kv_heads;
    size_t kb = planes * ctx->Lp * HD * (kv_dtype ? 1 : 2);
    std::vector<std::pair<uint8_t **, size_t>> want = {{&a.k, kb}, {&a.v, kb}};
    if (kv_dtype) {
        want.push_back({&a.ks, planes * ctx->Lp * 4 * 2});
        want.push_back({&a.vs, planes * ctx->Lp * 4 * 2});
    }
    for (auto &w : want) {
        void *p = nullptr;
        if (cudaMalloc(&p, w.second) != cudaSuccess) {
            cudaGetLastError();
            return bail(fail(nullptr, ZDEC_ERR_OOM, "cannot allocate the KV arena (%zu bytes for max_B=%d, max_L=%d)",
                             w.second, max_B, max_L));
        }
        ctx->arena_allocs.push_back(p);
        *w.first = (uint8_t *)p;
        ctx->arena_bytes += w.second;
        if (cudaMemsetAsync(p, 0, w.second, ctx->stream) != cudaSuccess)
            return bail(fail(nullptr, ZDEC_ERR_CUDA, "arena memset failed"));
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
        const int Kmax = std::max({H, F, ctx->qd});
        int lm_grid = n_groups(ctx->nrt_vocab) * 8;   // any cluster split of the LM head
        size_t w = 0;
        auto t = [&](size_t bytes) { size_t o = w; w = align_up(w + bytes, 256); return o; };
        size_t ox = t((size_t)Bm * H * 4), oqkv = t((size_t)Bm * ctx->qkv_ld * 4), oo2 = t((size_t)Bm * ctx->qd * 4);
        size_t oact = t((size_t)Bm * F * 4), olog = t((size_t)Bm * d.vocab * 4);
        size_t opart = t((size_t)Bm * d.n_kv_heads * 64 * 4 * (HD + 2) * 4);
        size_t oav = t((size_t)lm_grid * MAX_B * 4), oai = t((size_t)lm_grid * MAX_B * 4);
        size_t otk = t((size_t)Bm * d.n_kv_heads * 4);
        size_t orms = t((size_t)(n_groups(H / 16) + 1) * MAX_B * 4);
        auto plane = [&](int K) { return (size_t)(K / QK) * Bp * 256 * 2; };
        auto sums = [&](int K) { return (size_t)(K / QK) * Bp * 16 * 2; };
        size_t ox16 = t(plane(H)), ox16lo = t(plane(H)), osx = t(sums(H));
        size_t oo16 = t(plane(ctx->qd)), oo16lo = t(plane(ctx->qd)), oosx = t(sums(ctx->qd));
        size_t oa16 = t(plane(F)), oa16lo = t(plane(F)), oasx = t(sums(F));
        (void)Kmax;
        size_t otok = t(Bm * 4), opos = t(Bm * 4), oids = t(Bm * 4), olen = t(Bm * 4), ost = t(4);
        size_t oqf = t((size_t)Bm * d.n_q_heads * 32 * 16);
        ctx->ws_bytes = w;
        if (cudaMalloc(&ctx->ws, w) != cudaSuccess) {
            cudaGetLastError();
            return bail(fail(nullptr, ZDEC_ERR_OOM, "cannot allocate %zu bytes of workspace", w));
        }
        uint8_t *b = (uint8_t *)ctx->ws;
        ctx->x = (float *)(b + ox); ctx->qkv = (float *)(b + oqkv); ctx->o = (float *)(b + oo2);
        ctx->act = (float *)(b + oact); ctx->logits = (float *)(b + olog); ctx->part = (float *)(b + opart);
        ctx->amax_v = (float *)(b + oav); ctx->amax_i = (int *)(b + oai); ctx->tickets = (int *)(b + otk);
        ctx->rms_part = (float *)(b + orms);
        ctx->x16 = (__half *)(b + ox16); ctx->x16lo = (__half *)(b + ox16lo); ctx->sx = (__half *)(b + osx);
        ctx->o16 = (__half *)(b + oo16); ctx->o16lo = (__half *)(b + oo16lo); ctx->osx = (__half *)(b + oosx);
        ctx->a16 = (__half *)(b + oa16); ctx->a16lo = (__half *)(b + oa16lo); ctx->asx = (__half *)(b + oasx);
        ctx->tok_dev = (int32_t *)(b + otok); ctx->pos_dev = (int32_t *)(b + opos);
        ctx->ids_dev = (int32_t *)(b + oids); ctx->len_dev = (int32_t *)(b + olen);
        ctx->status = (uint32_t *)(b + ost);
        ctx->qfrag = (uint4 *)(b + oqf);
        if (cudaMemsetAsync(ctx->ws, 0, w, ctx->stream) != cudaSuccess)
            return bail(fail(nullptr, ZDEC_ERR_CUDA, "workspace memset failed"));
        if (cudaMallocHost(&ctx->pinned_io, 2 * Bm * sizeof(int32_t)) != cudaSuccess)
            return bail(fail(nullptr, ZDEC_ERR_OOM, "cannot allocate pinned staging"));
    }
    {
        // K splits of every projection for every kernel and batch class, from
        // the occupancy API (ZDEC_CS_MAX: largest split, default 16, a
        // non-portable cluster size)
        const int csmax = getenv("ZDEC_CS_MAX") ? std::max(1, std::min(16, atoi(getenv("ZDEC_CS_MAX")))) : 16;
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
                        groups[m], nsb[m], [&](int cs) { return gemm_cluster_slots(Bc, impl, epi[m], cs); }, csmax);
            }
        cudaGetLastError();
        if (getenv("ZDEC_PRINT_SPLITS"))   // impl, batch class: splits of qkv, o, gate/up, down, lm head
            for (int impl = 1; impl <= 3; impl++)
                for (int c = 0; c < 5; c++)
                    if (ctx->cs_tab[impl][c][0])
                        fprintf(stderr, "zdec splits impl %d B<=%d: %d %d %d %d %d\n", impl, CLASS_B[c],
                                ctx->cs_tab[impl][c][0], ctx->cs_tab[impl][c][1], ctx->cs_tab[impl][c][2],
                                ctx->cs_tab[impl][c][3], ctx->cs_tab[impl][c][4]);
    }
    if (attention_setup(kv_dtype) != cudaSuccess)
        return bail(fail(nullptr, ZDEC_ERR_CUDA, "attention smem attribute failed"));
    {
        zdec_status ss = step_configure(ctx);
        if (ss != ZDEC_OK) return bail(ss);
    }

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

extern "C" void zdec_destroy(zdec_ctx *ctx) {
    if (!ctx) return;
    cudaStreamSynchronize(ctx->stream);
    free_ctx(ctx);
}

extern "C" const char *zdec_last_error(const zdec_ctx *ctx) { return ctx ? ctx->err.c_str() : g_global_error.c_str(); }
extern "C" const char *zdec_last_global_error(void) { return g_global_error.c_str(); }

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
    const zdec_model_desc &d = ctx->d;
    size_t bytes = (size_t)d.n_layers * n_tokens * d.n_kv_heads * HD * 2;
    const uint16_t *kd = (const uint16_t *)k_f16, *vd = (const uint16_t *)v_f16;
    void *tmp = nullptr;
    if (!on_device) {
        if (cudaMalloc(&tmp, 2 * bytes) != cudaSuccess) {
            cudaGetLastError();
            return fail(ctx, ZDEC_ERR_OOM, "cannot stage %zu bytes of KV", 2 * bytes);
        }
        CK(cudaMemcpyAsync(tmp, k_f16, bytes, cudaMemcpyHostToDevice, ctx->stream));
        CK(cudaMemcpyAsync((uint8_t *)tmp + bytes, v_f16, bytes, cudaMemcpyHostToDevice, ctx->stream));
        kd = (const uint16_t *)tmp;
        vd = (const uint16_t *)((uint8_t *)tmp + bytes);
    }
    int t0 = ctx->len_host[seq];
    cudaError_t e = launch_kv_append(ctx->arena, seq, t0, n_tokens, kd, vd, ctx->stream);
    int32_t newlen = t0 + n_tokens;
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(ctx->len_dev + seq, &newlen, 4, cudaMemcpyHostToDevice, ctx->stream);
    if (!on_device) {
        cudaError_t e2 = cudaStreamSynchronize(ctx->stream);
        cudaFree(tmp);
        if (e == cudaSuccess) e = e2;
    } else if (e == cudaSuccess) {
        e = cudaStreamSynchronize(ctx->stream);   // the host length source is read asynchronously
    }
    if (e != cudaSuccess) return fail(ctx, ZDEC_ERR_CUDA, "append_kv: %s", cudaGetErrorString(e));
    ctx->len_host[seq] = newlen;
    return ZDEC_OK;
}

extern "C" zdec_status zdec_reset_seq(zdec_ctx *ctx, int seq) {
    if (!ctx) return fail(nullptr, ZDEC_ERR_ARG, "null context");
    if (seq < 0 || seq >= ctx->max_B) return fail(ctx, ZDEC_ERR_ARG, "seq %d out of range", seq);
    int32_t zero = 0;
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
// Attention split (cluster size, 1..16; ZDEC_ATT_CS forces one): the split
// of least modelled time over the B x n_kv clusters, waves x (chunks per CTA
// + 1 for the CTA's query load and merge) for a nominal 64 chunks per
// sequence, the waves from the occupancy API's co-resident clusters (which
// must each fit one GPC: 64 clusters of 6 Q8_0 CTAs fit at once, of 7 not).
static int attn_stages(const zdec_ctx *ctx, int B);
static int attn_cluster(const zdec_ctx *ctx, int B) {
    static const int forced = getenv("ZDEC_ATT_CS") ? atoi(getenv("ZDEC_ATT_CS")) : 0;
    if (forced >= 1 && forced <= 16) return forced;
    const int clusters = B * ctx->d.n_kv_heads, stages = attn_stages(ctx, B);
    int best = 1;
    double best_t = 1e30;
    for (int cs = 1; cs <= 16; cs++) {
        const int maxc = attention_max_clusters(ctx->kv_dtype, stages, cs);
        if (maxc <= 0) continue;
        const double t = (double)((clusters + maxc - 1) / maxc) * (64.0 / cs + 1.0);
        if (t < best_t - 1e-9) { best_t = t; best = cs; }
    }
    if (getenv("ZDEC_PRINT_SPLITS")) fprintf(stderr, "zdec attention B=%d: %d stages, split %d\n", B, stages, best);
    return best;
}

// Attention chunks in flight per CTA (ZDEC_ATT_STAGES overrides).  A deeper
// ring pays off only where the attention dominates the step; elsewhere its
// shared memory keeps the neighbouring projections' CTAs (which prefetch
// their weights) off the SMs.  Measured: batch of one, two stages; batch of
// eight, two for an fp16 cache (a third would drop to one CTA per SM) and
// three for Q8_0 (still three CTAs per SM).
static int attn_stages(const zdec_ctx *ctx, int B) {
    static const int env = getenv("ZDEC_ATT_STAGES") ? atoi(getenv("ZDEC_ATT_STAGES")) : 0;
    if (env >= 2) return std::min(env, ctx->kv_dtype ? 8 : 5);
    return (B > 4 && ctx->kv_dtype) ? 3 : 2;
}

static int pick_impl(const zdec_ctx *ctx, int B) {
    if (B > 4) return 2;
    if (ctx->gemm_impl == 1) return 1;
    if (ctx->gemm_impl == 2) return 2;
    if (ctx->gemm_impl == 3) return B == 1 ? 3 : 2;
    if (B == 1) return ctx->b1_impl;
    return B <= ctx->matvec_max_B ? 1 : 2;
}

// Enqueue the whole step for rows 0..B-1.  logits_out may be null.
static cudaError_t enqueue_step(zdec_ctx *ctx, int B, float *logits_out, bool pdl) {
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
    STEP(ZDEC_KERNEL_EMBED, launch_embed(ctx->embed, ctx->nsb_h, d.vocab, ctx->tok_dev, ctx->pos_dev,
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
    gp.pipe = gemm_pipe_mode();
    // Every projection takes its activation as fp16 hi + lo planes (~22 bits):
    // the new K/V rows are rounded and quantized, and over dozens of layers a
    // single fp16 operand would drift past the parity tolerance.
    auto operand = [&](__half *hi, __half *lo, __half *sums) { gp.x16 = hi; gp.x16lo = lo; gp.sx = sums; };
    auto matrix = [&](const uint8_t *W, int N, int nrt, int nsb, int cs) {
        gp.W = W; gp.N = N; gp.nrt = nrt; gp.nsb = nsb; gp.cs = cs;
        gp.pf_ptr = nullptr; gp.pf_bytes = 0;
    };
    // the next weight matrix to warm in L2 while a GEMM runs (capped so the
    // prefetched bytes and the running kernel's stream fit in L2 together)
    auto prefetch = [&](const uint8_t *W, int nrt, int nsb) {
        gp.pf_ptr = W;
        gp.pf_bytes = std::min(tile_bytes(nrt, nsb), ctx->prefetch_cap);
    };
    AttnParams ap{};
    ap.kv = ctx->arena;
    ap.nq = d.n_q_heads;
    ap.positions = ctx->pos_dev;
    ap.qkv = ctx->qkv;
    ap.qkv_ld = ctx->qkv_ld;
    ap.rope = ctx->rope;
    ap.append = 1;
    ap.cs = attn_cluster(ctx, B);
    ap.stages = attn_stages(ctx, B);
    ap.o = ctx->o;
    ap.o16 = ctx->o16;
    ap.o16lo = ctx->o16lo;
    ap.osx = ctx->osx;
    ap.oBp = Bp;
    ap.B = B;
    ap.max_L = ctx->max_L;
    ap.status = ctx->status;
    ap.q_frag = ctx->qfrag;   // written by the QKV projection's epilogue
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
        prefetch(lw.o, H / 16, ctx->nsb_q);
        gp.out = ctx->qkv; gp.ldo = ctx->qkv_ld;
        gp.q_frag = ctx->qfrag; gp.q_pos = ctx->pos_dev; gp.q_rope = ctx->rope; gp.q_heads = d.n_q_heads;
        STEP(ZDEC_KERNEL_GEMM_QKV, (gp.tl = tlk, launch_gemm(gp, EPI_STORE, impl, pdl, s)));
        gp.q_frag = nullptr;
        ap.layer = l;
        STEP(ZDEC_KERNEL_ATTENTION, (ap.tl = tlk, launch_attention(ap, pdl, s)));
        plain_input(ctx->o16, ctx->o16lo, ctx->osx);   // written by the attention combine
        matrix(lw.o, H, H / 16, ctx->nsb_q, split(MAT_O));
        prefetch(lw.gu, F / 8, ctx->nsb_h);
        gp.out = ctx->x; gp.ldo = H;
        gp.next_gain = lw.ffn_norm; gp.part_out = ctx->rms_part;
        gp.out16 = ctx->x16; gp.out16lo = ctx->x16lo; gp.out_sx = ctx->sx;
        STEP(ZDEC_KERNEL_GEMM_O, (gp.tl = tlk, launch_gemm(gp, EPI_RESID, impl, pdl, s)));
        normed_input(resid_groups);
        matrix(lw.gu, F, F / 8, ctx->nsb_h, split(MAT_GU));
        prefetch(lw.down, H / 16, ctx->nsb_f);
        gp.out = nullptr; gp.ldo = F;
        gp.out16 = ctx->a16; gp.out16lo = ctx->a16lo; gp.out_sx = ctx->asx;
        STEP(ZDEC_KERNEL_GEMM_GATEUP, (gp.tl = tlk, launch_gemm(gp, EPI_SWIGLU, impl, pdl, s)));
        plain_input(ctx->a16, ctx->a16lo, ctx->asx);   // written by the gate/up epilogue
        matrix(lw.down, H, H / 16, ctx->nsb_f, split(MAT_DOWN));
        if (l + 1 < d.n_layers) prefetch(ctx->L[l + 1].qkv, ctx->qkv_ld / 16, ctx->nsb_h);
        else prefetch(ctx->embed, ctx->nrt_vocab, ctx->nsb_h);
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
                                                 ctx->pos_dev, ctx->len_dev, ctx->status, pdl, s, tlk));
#undef STEP
    ctx->last_kernels = nk;
    ctx->last_splits = ap.cs;
    return cudaSuccess;
}

// The persistent kernel runs this step?
static bool use_persistent(const zdec_ctx *ctx, int B) {
    return ctx->engine == ZDEC_ENGINE_PERSISTENT && ctx->step_grid > 0 && B <= STEP_MAX_B;
}

// The whole step as the prep kernel + the persistent step kernel.
static cudaError_t enqueue_step_persistent(zdec_ctx *ctx, int B, float *logits_out) {
    const zdec_model_desc &d = ctx->d;
    StepParams p{};
    p.n_layers = d.n_layers;
    p.hidden = d.hidden;
    p.ffn = d.ffn;
    p.vocab = d.vocab;
    p.n_q = d.n_q_heads;
    p.n_kv = d.n_kv_heads;
    p.eps = d.rms_eps;
    p.layers = ctx->d_layers;
    p.embed = ctx->embed;
    p.lm = ctx->embed;
    p.final_norm = ctx->final_norm;
    p.rope = ctx->rope;
    p.kv = ctx->arena;
    p.max_L = ctx->max_L;
    p.B = B;
    p.tokens = ctx->tok_dev;
    p.positions = ctx->pos_dev;
    p.logits = logits_out;
    p.ids = ctx->ids_dev;
    p.capture = ctx->capture_dev_host ? ctx->s_capture : nullptr;
    p.x = ctx->x;
    p.u16 = ctx->x16; p.u16lo = ctx->x16lo; p.usx = ctx->sx;
    p.g16 = ctx->g16; p.g16lo = ctx->g16lo; p.gsx = ctx->gsx;
    p.o16 = ctx->o16; p.o16lo = ctx->o16lo; p.osx = ctx->osx;
    p.a16 = ctx->a16; p.a16lo = ctx->a16lo; p.asx = ctx->asx;
    p.rms_attn = ctx->rms_part;
    p.rms_ffn = ctx->s_rms_ffn;
    p.q = ctx->s_q;
    p.gpart = ctx->s_gpart;
    p.apart = ctx->s_apart;
    p.amax_val = ctx->amax_v;
    p.amax_idx = ctx->amax_i;
    p.cnt = ctx->s_cnt;
    p.n_cnt = ctx->s_ncnt;
    p.step_ok = ctx->s_ok;
    p.abort_flag = ctx->s_abort;
    p.status = ctx->status;
    p.slots = ctx->step_slots[B <= 4 ? 0 : 1];
    p.slot_bytes = step_slot_bytes(B);
    p.pf_items = ctx->step_pf_items;
    p.att_min_units = ctx->step_att_min;
    p.trace = ctx->trace_on ? ctx->trace : nullptr;
    cudaStream_t s = ctx->stream;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (ctx->prof) {
        cudaEventCreate(&e0);
        cudaEventCreate(&e1);
        cudaEventRecord(e0, s);
    }
    cudaError_t e = launch_step(p, ctx->step_grid, ctx->len_dev, s);
    if (ctx->prof) {
        cudaEventRecord(e1, s);
        ctx->prof->push_back(Launch{ZDEC_KERNEL_STEP, e0, e1});
    }
    if (e != cudaSuccess) return e;
    if (ctx->capture_dev_host)
        e = cudaMemcpyAsync(ctx->capture_dev_host, ctx->s_capture, (size_t)(d.n_layers + 1) * B * d.hidden * 4,
                            cudaMemcpyDeviceToHost, s);
    ctx->last_kernels = 2;
    ctx->last_splits = 0;
    return e;
}

static cudaError_t enqueue_any(zdec_ctx *ctx, int B, float *logits_out, bool pdl) {
    if (use_persistent(ctx, B)) {
        ctx->last_engine = ZDEC_ENGINE_PERSISTENT;
        return enqueue_step_persistent(ctx, B, logits_out);
    }
    ctx->last_engine = ZDEC_ENGINE_KERNELS;
    return enqueue_step(ctx, B, logits_out, pdl);
}

static zdec_status check_step_args(zdec_ctx *ctx, int B, const int32_t *tokens, const int32_t *positions,
                                   int32_t *ids) {
    if (!ctx) return fail(nullptr, ZDEC_ERR_ARG, "null context");
    if (B < 1 || B > ctx->max_B) return fail(ctx, ZDEC_ERR_ARG, "B=%d outside [1, %d]", B, ctx->max_B);
    if (!tokens || !positions || !ids) return fail(ctx, ZDEC_ERR_ARG, "null tokens/positions/ids");
    for (int b = 0; b < B; b++)
        if (ctx->len_host[b] + 1 > ctx->max_L)
            return fail(ctx, ZDEC_ERR_CAPACITY, "sequence %d is full (%d tokens)", b, ctx->max_L);
    if (ctx->engine == ZDEC_ENGINE_PERSISTENT && !use_persistent(ctx, B))
        return fail(ctx, ZDEC_ERR_UNSUPPORTED, "the persistent step kernel is unavailable for B=%d", B);
    return ZDEC_OK;
}

// Stage inputs: host pointers are validated and copied through pinned memory.
static zdec_status stage_inputs(zdec_ctx *ctx, int B, const int32_t *tokens, const int32_t *positions, bool host) {
    if (host) {
        for (int b = 0; b < B; b++) {
            if (positions[b] != ctx->len_host[b])
                return fail(ctx, ZDEC_ERR_POSITION, "positions[%d] = %d but sequence %d holds %d tokens", b,
                            positions[b], b, ctx->len_host[b]);
            if (tokens[b] < 0 || tokens[b] >= ctx->d.vocab)
                return fail(ctx, ZDEC_ERR_ARG, "tokens[%d] = %d outside the vocabulary", b, tokens[b]);
        }
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

extern "C" zdec_status zdec_decode_step(zdec_ctx *ctx, int B, const int32_t *tokens,
                                        const int32_t *positions, float *logits, int32_t *ids, int flags) {
    zdec_status st = check_step_args(ctx, B, tokens, positions, ids);
    if (st != ZDEC_OK) return st;
    const bool host = flags & ZDEC_STEP_HOST_IO;
    const bool eager = (flags & ZDEC_STEP_EAGER) || ctx->capture_dev_host || ctx->trace_on ||
                       (ctx->persistent_eager && use_persistent(ctx, B));
    st = stage_inputs(ctx, B, tokens, positions, host);
    if (st != ZDEC_OK) return st;
    float *lg = host ? (logits ? ctx->logits : nullptr) : logits;
    const int impl = use_persistent(ctx, B) ? 3 : pick_impl(ctx, B);
    if (eager) {
        CK(enqueue_any(ctx, B, lg, true));
    } else {
        auto key = std::make_tuple(B, (const void *)lg, impl);
        auto it = ctx->graphs.find(key);
        if (it == ctx->graphs.end()) {
            cudaGraph_t graph;
            CK(cudaStreamBeginCapture(ctx->stream, cudaStreamCaptureModeThreadLocal));
            cudaError_t e = enqueue_any(ctx, B, lg, true);
            cudaError_t e2 = cudaStreamEndCapture(ctx->stream, &graph);
            if ((e != cudaSuccess || e2 != cudaSuccess) && impl == 3) {
                // a cooperative launch that cannot be captured: run the persistent engine without graphs
                if (e2 == cudaSuccess) cudaGraphDestroy(graph);
                cudaGetLastError();
                ctx->persistent_eager = true;
                CK(enqueue_any(ctx, B, lg, true));
                goto launched;
            }
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
launched:
    if (host) {
        if (logits)
            CK(cudaMemcpyAsync(logits, ctx->logits, (size_t)B * ctx->d.vocab * 4, cudaMemcpyDeviceToHost, ctx->stream));
        CK(cudaMemcpyAsync(ids, ctx->ids_dev, B * 4, cudaMemcpyDeviceToHost, ctx->stream));
    } else {
        CK(cudaMemcpyAsync(ids, ctx->ids_dev, B * 4, cudaMemcpyDeviceToDevice, ctx->stream));
    }
    for (int b = 0; b < B; b++) ctx->len_host[b]++;
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
        return fail(ctx, ZDEC_ERR_DEVICE, "device check failed (status 0x%x:%s%s)", st,
                    (st & STATUS_POSITION) ? " position != cached length" : "",
                    (st & STATUS_TOKEN) ? " token outside the vocabulary" : "");
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
    info->arena_bytes = ctx->arena_bytes;
    info->workspace_bytes = ctx->ws_bytes;
    info->kv_bytes_per_token = (size_t)ctx->d.n_layers * ctx->d.n_kv_heads * HD * 2 * (ctx->kv_dtype ? 1 : 2) +
                               (ctx->kv_dtype ? (size_t)ctx->d.n_layers * ctx->d.n_kv_heads * 4 * 2 * 2 : 0);
    info->kernels_per_step = ctx->last_kernels;
    info->attn_splits = ctx->last_splits;
    info->matvec_max_B = ctx->matvec_max_B;
    info->engine = ctx->last_engine;
    info->step_ctas = ctx->step_grid;
    return ZDEC_OK;
}

extern "C" zdec_status zdec_set_trace(zdec_ctx *ctx, int on) {
    if (!ctx) return fail(nullptr, ZDEC_ERR_ARG, "null context");
    CK(cudaStreamSynchronize(ctx->stream));
    if (!on) {
        cudaFree(ctx->trace);
        cudaFree(ctx->ktl);
        cudaFreeHost(ctx->ktl_init);
        ctx->trace = nullptr;
        ctx->ktl = nullptr;
        ctx->ktl_init = nullptr;
        ctx->trace_entries = ctx->ktl_entries = 0;
        ctx->trace_on = false;
        return ZDEC_OK;
    }
    if (ctx->trace_on) return ZDEC_OK;
    if (ctx->step_grid > 0) {   // persistent engine: [ctas][phases][8]
        const size_t n = (size_t)ctx->step_grid * (2 + 5 * ctx->d.n_layers) * 8;
        if (cudaMalloc(&ctx->trace, n * 8) != cudaSuccess) {
            cudaGetLastError();
            return fail(ctx, ZDEC_ERR_OOM, "cannot allocate the step trace");
        }
        CK(cudaMemsetAsync(ctx->trace, 0, n * 8, ctx->stream));
        ctx->trace_entries = n;
    }
    // kernel engine: [launches][8] = (first start, first past the wait, last end, kind, milestones)
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
    const bool pers = ctx->last_engine == ZDEC_ENGINE_PERSISTENT;
    *n = !ctx->trace_on ? 0 : (pers ? ctx->trace_entries : ctx->ktl_entries);
    if (!ctx->trace_on || !out_host || *n == 0) return ZDEC_OK;   // size query
    if (cap < *n) return fail(ctx, ZDEC_ERR_ARG, "trace needs %zu entries", *n);
    CK(cudaStreamSynchronize(ctx->stream));
    CK(cudaMemcpy(out_host, pers ? ctx->trace : ctx->ktl, *n * 8, cudaMemcpyDeviceToHost));
    if (!pers)
        for (size_t i = 0; i < *n / 8; i++) out_host[8 * i + 3] = i < ctx->ktl_kinds.size() ? ctx->ktl_kinds[i] : 0;
    return ZDEC_OK;
}

extern "C" zdec_status zdec_set_engine(zdec_ctx *ctx, int engine) {
    if (!ctx) return fail(nullptr, ZDEC_ERR_ARG, "null context");
    if (engine < ZDEC_ENGINE_AUTO || engine > ZDEC_ENGINE_PERSISTENT) return fail(ctx, ZDEC_ERR_ARG, "bad engine %d", engine);
    if (engine == ZDEC_ENGINE_PERSISTENT && ctx->step_grid == 0)
        return fail(ctx, ZDEC_ERR_UNSUPPORTED, "the persistent step kernel is unavailable on this device/model");
    ctx->engine = engine;
    return ZDEC_OK;
}

extern "C" zdec_status zdec_profile_step(zdec_ctx *ctx, int B, const int32_t *tokens_dev,
                                         const int32_t *positions_dev, float *logits_dev, int32_t *ids_dev,
                                         int *kind, float *ms, int cap, int *n) {
    zdec_status st = check_step_args(ctx, B, tokens_dev, positions_dev, ids_dev);
    if (st != ZDEC_OK) return st;
    if (!n || (cap > 0 && (!kind || !ms))) return fail(ctx, ZDEC_ERR_ARG, "null output");
    st = stage_inputs(ctx, B, tokens_dev, positions_dev, false);
    if (st != ZDEC_OK) return st;
    std::vector<Launch> launches;
    ctx->prof = &launches;
    cudaError_t e = enqueue_any(ctx, B, logits_dev, false);
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
    for (int b = 0; b < B; b++) ctx->len_host[b]++;
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
    if (ctx->kv_dtype && (!ks || !vs)) return fail(ctx, ZDEC_ERR_ARG, "Q8_0 read needs scale buffers");
    if (seq < 0 || seq >= ctx->max_B || layer < 0 || layer >= ctx->d.n_layers || t0 < 0 || n < 0 ||
        t0 + n > ctx->max_L)
        return fail(ctx, ZDEC_ERR_ARG, "range out of bounds");
    if (n == 0) return ZDEC_OK;
    const int nkv = ctx->d.n_kv_heads;
    size_t es = ctx->kv_dtype ? 1 : 2;
    size_t kb = (size_t)n * nkv * HD * es, sb = ctx->kv_dtype ? (size_t)n * nkv * 4 * 2 : 0;
    uint8_t *buf = nullptr;
    if (cudaMalloc(&buf, 2 * kb + 2 * sb + 16) != cudaSuccess) { cudaGetLastError(); return fail(ctx, ZDEC_ERR_OOM, "debug buffer"); }
    uint16_t *dks = sb ? (uint16_t *)(buf + 2 * kb) : nullptr, *dvs = sb ? (uint16_t *)(buf + 2 * kb + sb) : nullptr;
    cudaError_t e = launch_kv_read(ctx->arena, seq, layer, t0, n, buf, buf + kb, dks, dvs, ctx->stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(k, buf, kb, cudaMemcpyDeviceToHost, ctx->stream);
    if (e == cudaSuccess) e = cudaMemcpyAsync(v, buf + kb, kb, cudaMemcpyDeviceToHost, ctx->stream);
    if (e == cudaSuccess && sb) e = cudaMemcpyAsync(ks, dks, sb, cudaMemcpyDeviceToHost, ctx->stream);
    if (e == cudaSuccess && sb) e = cudaMemcpyAsync(vs, dvs, sb, cudaMemcpyDeviceToHost, ctx->stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(ctx->stream);
    cudaFree(buf);
    if (e != cudaSuccess) return fail(ctx, ZDEC_ERR_CUDA, "kv read: %s", cudaGetErrorString(e));
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
    AttnParams ap{};
    ap.kv = ctx->arena;
    ap.layer = layer;
    ap.nq = ctx->d.n_q_heads;
    ap.positions = ctx->pos_dev;
    ap.qkv = ctx->qkv;
    ap.qkv_ld = ctx->qkv_ld;
    ap.rope = ctx->rope;
    ap.append = 0;
    ap.cs = attn_cluster(ctx, B);
    ap.o = ctx->o;
    ap.o16 = ctx->o16;
    ap.o16lo = ctx->o16lo;
    ap.osx = ctx->osx;
    ap.oBp = ctx->Bp_max;
    ap.B = B;
    ap.max_L = ctx->max_L;
    ap.status = ctx->status;
    CK(launch_attention(ap, false, ctx->stream));
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
    gp.pipe = gemm_pipe_mode();
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
