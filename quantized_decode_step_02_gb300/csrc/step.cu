// step.cu -- one decode step as a single persistent, cooperative kernel.
//
// Why one kernel: at batch one a step is ~180 dependent phases (per layer the
// QKV projection, attention, O, gate/up and down) whose weights take 1-10 us
// each to stream at full HBM rate, so per-kernel launch, ramp-up and drain
// cost as much as the bytes.  Here every SM runs the whole step and the only
// thing a phase waits for is its activations: the weight bytes of the next
// phase (and the KV history of the next attention) do not depend on this
// step's data, so each CTA's producer warp keeps streaming them into a ring
// of shared-memory slots while the consumers wait for the activations ("The
// weight read is the only term that does not scale": the stream runs
// regardless of where the data dependencies are).
//
// CTA = 8 consumer warps + 1 producer warp; two CTAs per SM; grid = 2 x SMs,
// launched cooperatively so every CTA is resident.
//
// Work split.  Every GEMM phase is a list of items (group, super-block): the
// 18,432-byte bulk copy of the group's 8 tile blocks for that super-block (one
// tile block per consumer warp) plus that super-block's activation rows.  The
// items of a phase are cut into equal contiguous ranges, one per CTA, so a
// group's K range may be split over consecutive CTAs ("pieces").  A piece's
// partial tile goes to global memory; the CTA that completes a group's last
// piece (a counter per group) sums all pieces in CTA order -- fixed order, so
// the result does not depend on timing -- and runs the group's epilogue.
// Attention items are 32-token units of one (sequence, kv head), cut the same
// way; partial (max, sum, output) states merge the same way.
//
// Dependencies are counters in global memory, incremented after a group's
// (or a head's) epilogue has written its outputs: QKV of head g -> attention
// of head g; all attention heads -> O; all O groups -> gate/up; all gate/up
// groups -> down; all down groups -> next layer's QKV (and the LM head).  The
// producer issues an item's weight copy as soon as its slot is free and the
// activation copy once the phase's counter is complete.  Every wait is
// bounded: on expiry the kernel sets STATUS_TIMEOUT and a global abort flag,
// and every CTA winds down (the producer first waits for its copies).
#include "attn_core.cuh"
#include "gemm_core.cuh"
#include "tiles.cuh"

namespace zdec {

namespace {

constexpr int CW = 8;                      // consumer warps per CTA
constexpr int CTHREADS = CW * 32;
constexpr int STEP_THREADS = CTHREADS + 32;
constexpr long long WAIT_LIMIT = 1LL << 32;   // clock cycles, ~2 s
constexpr int QKV_PER_HEAD = GROUP + 2;     // q groups of a kv head + its k and v groups

// ------------------------------------------------------------ PTX helpers
__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ int ld_acquire(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}
__device__ __forceinline__ void mbar_arrive_n(uint64_t *bar, uint32_t n) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(n) : "memory");
}

// ------------------------------------------------------------ model dims
struct Dims {
    int L, H, F, V, nq, nkv;
    int nsb_h, nsb_f;
    int nrt_qkv, nrt_o, nrt_gu, nrt_down, nrt_lm;
    int g_qkv, g_o, g_gu, g_down, g_lm;
    // counter indices
    int c_lm, pc_base, pc_stride, pc_lm, n_cnt;
};
__host__ __device__ inline Dims make_dims(int L, int H, int F, int V, int nq, int nkv) {
    Dims d;
    d.L = L; d.H = H; d.F = F; d.V = V; d.nq = nq; d.nkv = nkv;
    d.nsb_h = H / QK;
    d.nsb_f = F / QK;
    d.nrt_qkv = (nq + 2 * nkv) * (HD / 16);
    d.nrt_o = H / 16;
    d.nrt_gu = F / 8;
    d.nrt_down = H / 16;
    d.nrt_lm = (V + 15) / 16;
    d.g_qkv = n_groups(d.nrt_qkv);
    d.g_o = n_groups(d.nrt_o);
    d.g_gu = n_groups(d.nrt_gu);
    d.g_down = n_groups(d.nrt_down);
    d.g_lm = n_groups(d.nrt_lm);
    d.c_lm = 1 + L * (nkv + 4);
    d.pc_base = d.c_lm + 1;
    d.pc_stride = d.g_qkv + d.g_o + d.g_gu + d.g_down + STEP_MAX_B * nkv;
    d.pc_lm = d.pc_base + L * d.pc_stride;
    d.n_cnt = d.pc_lm + d.g_lm;
    return d;
}
// completion counters: 0 = embedding items; per layer qkv heads, att, o, gu, down
__device__ __forceinline__ int c_qkvh(const Dims &d, int l, int g) { return 1 + l * (d.nkv + 4) + g; }
__device__ __forceinline__ int c_att(const Dims &d, int l) { return 1 + l * (d.nkv + 4) + d.nkv; }
__device__ __forceinline__ int c_o(const Dims &d, int l) { return c_att(d, l) + 1; }
__device__ __forceinline__ int c_gu(const Dims &d, int l) { return c_att(d, l) + 2; }
__device__ __forceinline__ int c_down(const Dims &d, int l) { return c_att(d, l) + 3; }

enum PhaseKind : int { PK_EMBED = 0, PK_QKV, PK_ATT, PK_O, PK_GU, PK_DOWN, PK_LM };

struct Phase {
    int kind, layer;
    int U;                          // items
    int G;                          // CTAs sharing them (the first G of the grid)
    // GEMM
    const uint8_t *W;
    int nsb, nrt;
    const __half *ihi, *ilo, *isx;  // input planes
    int gate, target;               // counter index and count that release the inputs
    int pc;                         // first piece counter of the phase
};

// Per-CTA shared state that every thread reads.
struct StepShared {
    int units[STEP_MAX_B + 1];      // prefix sums of 32-token units per sequence
    int pos[STEP_MAX_B];
    float r[STEP_MAX_B];            // RMSNorm scales of the current phase
    int last;                       // broadcast: this CTA completes the piece's group
    int abort;                      // monotonic: stop
};

__device__ __forceinline__ int n_phases(const Dims &d) { return 2 + 5 * d.L; }

__device__ Phase make_phase(const StepParams &p, const Dims &d, const StepShared &sh, int ph) {
    Phase f{};
    f.G = gridDim.x;
    if (ph == 0) { f.kind = PK_EMBED; f.U = p.B * (d.H / 128); return f; }
    if (ph == 1 + 5 * d.L) {
        f.kind = PK_LM; f.layer = d.L;
        f.W = p.lm; f.nsb = d.nsb_h; f.nrt = d.nrt_lm; f.U = d.g_lm * d.nsb_h;
        f.ihi = p.u16; f.ilo = p.u16lo; f.isx = p.usx;
        f.gate = c_down(d, d.L - 1); f.target = d.g_down;
        f.pc = d.pc_lm;
        return f;
    }
    const int l = (ph - 1) / 5, k = (ph - 1) % 5;
    const StepLayerW &w = p.layers[l];
    const int pcl = d.pc_base + l * d.pc_stride;
    f.layer = l;
    switch (k) {
        case 0:
            f.kind = PK_QKV; f.W = w.qkv; f.nsb = d.nsb_h; f.nrt = d.nrt_qkv; f.U = d.g_qkv * d.nsb_h;
            f.ihi = p.u16; f.ilo = p.u16lo; f.isx = p.usx;
            if (l == 0) { f.gate = 0; f.target = p.B * (d.H / 128); }
            else { f.gate = c_down(d, l - 1); f.target = d.g_down; }
            f.pc = pcl;
            break;
        case 1:
            f.kind = PK_ATT; f.U = d.nkv * sh.units[p.B];
            f.G = max(1, min(f.G, f.U / max(1, p.att_min_units)));
            f.gate = -1; f.target = 0;
            f.pc = pcl + d.g_qkv + d.g_o + d.g_gu + d.g_down;
            break;
        case 2:
            f.kind = PK_O; f.W = w.o; f.nsb = d.nsb_h; f.nrt = d.nrt_o; f.U = d.g_o * d.nsb_h;
            f.ihi = p.o16; f.ilo = p.o16lo; f.isx = p.osx;
            f.gate = c_att(d, l); f.target = p.B * d.nkv;
            f.pc = pcl + d.g_qkv;
            break;
        case 3:
            f.kind = PK_GU; f.W = w.gu; f.nsb = d.nsb_h; f.nrt = d.nrt_gu; f.U = d.g_gu * d.nsb_h;
            f.ihi = p.g16; f.ilo = p.g16lo; f.isx = p.gsx;
            f.gate = c_o(d, l); f.target = d.g_o;
            f.pc = pcl + d.g_qkv + d.g_o;
            break;
        default:
            f.kind = PK_DOWN; f.W = w.down; f.nsb = d.nsb_f; f.nrt = d.nrt_down; f.U = d.g_down * d.nsb_f;
            f.ihi = p.a16; f.ilo = p.a16lo; f.isx = p.asx;
            f.gate = c_gu(d, l); f.target = d.g_gu;
            f.pc = pcl + d.g_qkv + d.g_o + d.g_gu;
            break;
    }
    return f;
}

// Equal contiguous ranges of U items over G CTAs; owner of item x.
__device__ __forceinline__ int range_lo(int U, int G, int c) { return (int)((long long)c * U / G); }
__device__ __forceinline__ int owner_of(int U, int G, int x) { return (int)(((long long)(x + 1) * G - 1) / U); }

// Attention item x -> (sequence b, kv head g, unit u, units of b).
__device__ __forceinline__ void att_item(const StepShared &sh, int nkv, int B, int x, int &b, int &g, int &u,
                                         int &nu) {
    b = 0;
    while (b + 1 < B && nkv * sh.units[b + 1] <= x) b++;
    nu = sh.units[b + 1] - sh.units[b];
    const int r = x - nkv * sh.units[b];
    g = r / nu;
    u = r % nu;
}

// ------------------------------------------------------------ ring plan
struct Copy { const void *src; uint32_t dst, bytes; };
struct Plan {
    int na, nb;
    Copy a[4], b[4];
    uint32_t total;
    int gate, target;
};

template <int KVT>
__device__ void plan_item(const StepParams &p, const Dims &d, const StepShared &sh, const Phase &f, int x,
                          const StageLayout &lay, Plan &pl) {
    pl.na = pl.nb = 0;
    pl.total = 0;
    pl.gate = -1;
    pl.target = 0;
    if (f.kind != PK_ATT) {
        const int grp = x / f.nsb, sb = x % f.nsb;
        pl.a[0] = {f.W + ((size_t)grp * f.nsb + sb) * GROUP_BYTES, 0u, (uint32_t)GROUP_BYTES};
        pl.na = 1;
        const uint32_t ab = (uint32_t)p.B * 512u, sbb = (uint32_t)p.B * 32u;
        pl.b[0] = {f.ihi + (size_t)sb * p.B * 256, lay.hi, ab};
        pl.b[1] = {f.ilo + (size_t)sb * p.B * 256, lay.lo, ab};
        pl.b[2] = {f.isx + (size_t)sb * p.B * 16, lay.sums, sbb};
        pl.nb = 3;
        pl.total = GROUP_BYTES + 2 * ab + sbb;
        pl.gate = f.gate;
        pl.target = f.target;
        return;
    }
    int b, g, u, nu;
    att_item(sh, d.nkv, p.B, x, b, g, u, nu);
    const size_t pi = ((size_t)b * d.L + f.layer) * d.nkv + g;
    const size_t Lp = p.kv.Lp;
    Copy c[4];
    int n;
    if (KVT == 0) {
        c[0] = {p.kv.k + pi * Lp * 256 + (size_t)u * 8192, 0u, 8192u};
        c[1] = {p.kv.v + pi * Lp * 256 + (size_t)u * 8192, 8192u, 8192u};
        n = 2;
        pl.total = 16384;
    } else {
        c[0] = {p.kv.k + pi * Lp * 128 + (size_t)u * 4096, 0u, 4096u};
        c[1] = {p.kv.ks + pi * Lp * 8 + (size_t)u * 256, 4096u, 256u};
        c[2] = {p.kv.v + pi * Lp * 128 + (size_t)u * 4096, 4352u, 4096u};
        c[3] = {p.kv.vs + pi * Lp * 8 + (size_t)u * 256, 8448u, 256u};
        n = 4;
        pl.total = 8704;
    }
    if (u == nu - 1) {   // holds this step's token: wait for the head's k/v append
        for (int i = 0; i < n; i++) pl.b[i] = c[i];
        pl.nb = n;
        pl.gate = c_qkvh(d, f.layer, g);
        pl.target = QKV_PER_HEAD;
    } else {
        for (int i = 0; i < n; i++) pl.a[i] = c[i];
        pl.na = n;
    }
}

// Iterates this CTA's items over all ring phases (everything but the embedding).
struct Cursor {
    int ph, x, hi;
    Phase f;
};
__device__ void cursor_seek(const StepParams &p, const Dims &d, const StepShared &sh, Cursor &c, int ph) {
    const int cta = blockIdx.x, NPH = n_phases(d);
    for (; ph < NPH; ph++) {
        c.f = make_phase(p, d, sh, ph);
        if (c.f.kind == PK_EMBED || cta >= c.f.G) continue;
        c.x = range_lo(c.f.U, c.f.G, cta);
        c.hi = range_lo(c.f.U, c.f.G, cta + 1);
        if (c.x < c.hi) break;
    }
    c.ph = ph;
}
__device__ __forceinline__ bool cursor_valid(const Dims &d, const Cursor &c) { return c.ph < n_phases(d); }
__device__ __forceinline__ void cursor_next(const StepParams &p, const Dims &d, const StepShared &sh, Cursor &c) {
    if (++c.x >= c.hi) cursor_seek(p, d, sh, c, c.ph + 1);
}

// Phase timeline (optional): trace[(cta * phases + ph) * 8 + k] = %globaltimer
// (ns).  k: 0 the consumers enter the phase, 1 its inputs are released (gate
// passed), 2 the first item has landed, 3 the last item is consumed, 4 the
// phase's epilogues are done, 5 producer: first copy of the phase issued,
// 6 producer: first activation (gated) copy issued, 7 items of the phase.
__device__ __forceinline__ unsigned long long gtime() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void trace_at(const StepParams &p, int ph, int k, unsigned long long v) {
    p.trace[((size_t)blockIdx.x * (2 + 5 * p.n_layers) + ph) * 8 + k] = v;
}
__device__ __forceinline__ void trace(const StepParams &p, int ph, int k) {
    if (p.trace && threadIdx.x == 0) trace_at(p, ph, k, gtime());
}

__device__ __forceinline__ void raise_abort(const StepParams &p) {
    atomicOr(p.status, STATUS_TIMEOUT);
    atomicExch(p.abort_flag, 1);
}
__device__ __forceinline__ bool aborted(const StepParams &p) {
    return *reinterpret_cast<volatile const int *>(p.abort_flag) != 0;
}

// -------------------------------------------------------------- producer
template <int KVT>
__device__ void producer(const StepParams &p, const Dims &d, const StepShared &sh, uint8_t *ring,
                         uint64_t *full, uint64_t *empty, const StageLayout &lay) {
    const int S = p.slots;
    const uint32_t SB = (uint32_t)p.slot_bytes;
    Cursor ca, cb, cp;
    cursor_seek(p, d, sh, ca, 0);
    cb = ca;
    cp = ca;
    uint32_t issued = 0, done_b = 0, pf_done = 0;
    int traced_a = -1, traced_b = -1;
    int ok_gate = -2, ok_target = 0;   // last gate seen complete
    long long t_idle = clock64();
    int spins = 0;
    bool abort = false;
    Plan pl;
    while (true) {
        bool prog = false;
        if (cursor_valid(d, ca)) {
            const uint32_t slot = issued % S, k = issued / S;
            if (k == 0 || mbar_test(&empty[slot], (k - 1) & 1u)) {
                if (p.trace && ca.ph != traced_a) {
                    trace_at(p, ca.ph, 5, gtime());
                    trace_at(p, ca.ph, 7, (unsigned long long)(ca.hi - ca.x));
                    traced_a = ca.ph;
                }
                plan_item<KVT>(p, d, sh, ca.f, ca.x, lay, pl);
                uint8_t *dst = ring + (size_t)slot * SB;
                mbar_expect_tx(&full[slot], pl.total);
                for (int i = 0; i < pl.na; i++) bulk_g2s(dst + pl.a[i].dst, pl.a[i].src, pl.a[i].bytes, &full[slot]);
                issued++;
                cursor_next(p, d, sh, ca);
                prog = true;
            }
        }
        if (done_b < issued) {
            plan_item<KVT>(p, d, sh, cb.f, cb.x, lay, pl);
            bool go = pl.nb == 0;
            if (!go) {
                if (pl.gate == ok_gate && pl.target <= ok_target) go = true;
                else if (ld_acquire(p.cnt + pl.gate) >= pl.target) {
                    ok_gate = pl.gate;
                    ok_target = pl.target;
                    go = true;
                }
                if (go) fence_proxy_async();
            }
            if (go) {
                if (p.trace && pl.nb && cb.ph != traced_b) {
                    trace_at(p, cb.ph, 6, gtime());
                    traced_b = cb.ph;
                }
                uint8_t *dst = ring + (size_t)(done_b % S) * SB;
                for (int i = 0; i < pl.nb; i++)
                    bulk_g2s(dst + pl.b[i].dst, pl.b[i].src, pl.b[i].bytes, &full[done_b % S]);
                done_b++;
                cursor_next(p, d, sh, cb);
                prog = true;
            }
        } else if (!cursor_valid(d, ca)) {
            break;
        }
        // L2 prefetch of the weight (and history) bytes of the next items:
        // the HBM stream runs ahead of the ring by pf_items items, so it keeps
        // going while the consumers wait for a phase's activations
        if (p.pf_items > 0 && cursor_valid(d, cp) && pf_done < issued + (uint32_t)p.pf_items) {
            if (pf_done >= issued) {
                plan_item<KVT>(p, d, sh, cp.f, cp.x, lay, pl);
                for (int i = 0; i < pl.na; i++) prefetch_l2(pl.a[i].src, pl.a[i].bytes);
                prog = true;
            }
            pf_done++;
            cursor_next(p, d, sh, cp);
        }
        if (prog) {
            t_idle = clock64();
            spins = 0;
            continue;
        }
        if (++spins > 8) __nanosleep(64);
        if ((spins & 15) == 0) {
            if (aborted(p)) { abort = true; break; }
            if (clock64() - t_idle > WAIT_LIMIT) { raise_abort(p); abort = true; break; }
        }
    }
    if (!abort) return;
    // wind down: complete every issued slot (the data is not used any more),
    // then wait for the copies so none lands after the CTA has exited
    while (done_b < issued) {
        plan_item<KVT>(p, d, sh, cb.f, cb.x, lay, pl);
        uint8_t *dst = ring + (size_t)(done_b % S) * SB;
        for (int i = 0; i < pl.nb; i++) bulk_g2s(dst + pl.b[i].dst, pl.b[i].src, pl.b[i].bytes, &full[done_b % S]);
        done_b++;
        cursor_next(p, d, sh, cb);
    }
    const uint32_t first = issued > (uint32_t)S ? issued - S : 0;
    const long long t0 = clock64();
    for (uint32_t i = first; i < issued; i++)
        while (!mbar_try_wait(&full[i % S], (i / S) & 1u))
            if (clock64() - t0 > WAIT_LIMIT) return;
}

// ------------------------------------------------------------ consumers
struct Ring {
    uint8_t *base;
    uint64_t *full, *empty;
    int S;
    uint32_t SB;
    __device__ __forceinline__ uint8_t *slot(uint32_t it) const { return base + (size_t)(it % S) * SB; }
};

// Bounded wait for item `it` to land (all lanes of the warp).  After an
// abort nothing waits any more: the consumers run through the rest of the
// step on whatever the buffers hold, so every warp still meets every
// barrier, and the kernel ends; the step's status reports the failure.
// A parity wait only tells two consecutive phases of a slot apart, so a
// consumer may wait for fill k of a slot only once fill k-1 has landed.  The
// GEMM consumers take every item in order; the attention's warp pairs take
// items round-robin over P pairs with P dividing the slot count, so every
// fill of a slot goes to the same pair, which has consumed the previous one.
__device__ __forceinline__ void wait_item(const StepParams &p, const Ring &r, uint32_t it, StepShared &sh) {
    uint64_t *bar = &r.full[it % r.S];
    const uint32_t par = (it / r.S) & 1u;
    if (sh.abort || mbar_try_wait(bar, par)) return;
    const long long t0 = clock64();
    int n = 0;
    while (!mbar_try_wait(bar, par)) {
        if ((++n & 15) == 0) {
            if (sh.abort || aborted(p)) { sh.abort = 1; return; }
            if (clock64() - t0 > WAIT_LIMIT) { raise_abort(p); sh.abort = 1; return; }
        }
    }
}
__device__ __forceinline__ void release_item(const Ring &r, uint32_t it, uint32_t count) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive_n(&r.empty[it % r.S], count);
}

// Thread 0 waits until counter `c` reaches `target`; warp 0 then computes the
// RMSNorm scales from `rms` (null: none).  Ends with a consumer barrier.
__device__ void gate_and_norm(const StepParams &p, StepShared &sh, int c, int target, const float *rms, int K) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0) {
        if (lane == 0 && c >= 0 && !sh.abort) {
            const long long t0 = clock64();
            int n = 0;
            while (ld_acquire(p.cnt + c) < target) {
                if ((++n & 15) == 0) {
                    if (aborted(p)) { sh.abort = 1; break; }
                    if (clock64() - t0 > WAIT_LIMIT) { raise_abort(p); sh.abort = 1; break; }
                }
                __nanosleep(32);
            }
        }
        __syncwarp();
        if (rms)
            for (int b = 0; b < p.B; b++) {
                float ss = 0.0f;
                for (int i = lane; i < K / 128; i += 32) ss += __ldcg(rms + i * MAX_B + b);
                for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(FULL, ss, o);
                if (lane == 0) sh.r[b] = 1.0f / sqrtf(ss / (float)K + p.eps);
            }
    }
    cbar();
}

// After a group's epilogue stores: make them visible (also to the bulk-copy
// engine) and count the group as done.
__device__ __forceinline__ void publish(const StepParams &p, int c) {
    fence_proxy_async();
    cbar();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(p.cnt + c, 1);
    }
}

// Write a piece partial, count it; returns true in the CTA that completes the
// item (it then reads all pieces).  n_pieces > 1.
__device__ bool piece_arrive(const StepParams &p, StepShared &sh, int counter, int n_pieces) {
    __threadfence();
    cbar();
    if (threadIdx.x == 0) {
        const int old = atomicAdd(p.cnt + counter, 1);
        sh.last = old == n_pieces - 1;
        if (sh.last) __threadfence();
    }
    cbar();
    return sh.last != 0;
}

// ---- embedding: x = E[token]; u planes = attn_norm[0] * x; x^2 partials
__device__ void embed_phase(const StepParams &p, const Dims &d, StepShared &sh, float *scr) {
    const int G = gridDim.x, t = threadIdx.x;
    const int per = d.H / 128;
    const float *gain = p.layers[0].attn_norm;
    for (int item = blockIdx.x; item < p.B * per; item += G) {
        const int b = item / per, i = item % per;
        const int tok = p.tokens[b];
        float w = 0.0f;
        if (t < 128) {
            const int k = 128 * (i & 1) + t, sb = i >> 1;
            const uint8_t *tile = p.embed + tile_offset(tok >> 4, sb, d.nsb_h);
            uint16_t dbits, mbits;
            int sc[8], m[8];
            tile_row_fields(tile, tok & 15, dbits, mbits, sc, m);
            const int j = k >> 5;
            w = dq_value(__half2float(__ushort_as_half(dbits)), sc[j], __half2float(__ushort_as_half(mbits)), m[j],
                         tile_q(tile, tok & 15, k));
            p.x[(size_t)b * d.H + 128 * i + t] = w;
            if (p.capture) p.capture[(size_t)b * d.H + 128 * i + t] = w;
            scr[t] = w;
        }
        cbar();
        if (t < 16) {   // chunk t of 8 values
            float yy[8], part = 0.0f, sq = 0.0f;
            const int r0 = 128 * i + 8 * t;
#pragma unroll
            for (int e = 0; e < 8; e++) {
                const float xv = scr[8 * t + e];
                sq = fmaf(xv, xv, sq);
                yy[e] = xv * gain[r0 + e];
                part += yy[e];
            }
            store_act8(p.u16, p.u16lo, act_chunk(r0 >> 8, b, (r0 & 255) >> 3, p.B), yy);
            part += __shfl_xor_sync(0xFFFFu, part, 1);
            part += __shfl_xor_sync(0xFFFFu, part, 2);
            if ((t & 3) == 0) store_sum(p.usx, r0 >> 8, b, (r0 & 255) >> 5, p.B, part);
            sq += __shfl_xor_sync(0xFFFFu, sq, 1);
            sq += __shfl_xor_sync(0xFFFFu, sq, 2);
            sq += __shfl_xor_sync(0xFFFFu, sq, 4);
            sq += __shfl_xor_sync(0xFFFFu, sq, 8);
            if (t == 0) p.rms_attn[i * MAX_B + b] = sq;
        }
        publish(p, 0);
    }
}

// ---- GEMM epilogues over a whole group; y: rows warp*16 + g + 8r, batch col 4nt + tig
template <int NT>
__device__ void to_smem(const StepParams &p, float *sy, const float (&y)[NT][2], bool scale, const StepShared &sh) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT; nt++) {
        const int b = 4 * nt + tig;
        if (b < p.B)
#pragma unroll
            for (int r = 0; r < 2; r++) sy[b * 128 + warp * 16 + g + 8 * r] = scale ? y[nt][r] * sh.r[b] : y[nt][r];
    }
}

template <int KVT>
__device__ void qkv_epilogue(const StepParams &p, const Dims &d, const StepShared &sh, int l, int grp, float *sy) {
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const float qscale = 0.08838834764831845f;   // 1/sqrt(128)
    int head;
    if (grp < d.nq) {   // query head: rotate, scale
        head = grp / GROUP;
        for (int task = t; task < p.B * 64; task += CTHREADS) {
            const int b = task >> 6, i = task & 63;
            const float2 cs = p.rope[(size_t)sh.pos[b] * 64 + i];
            const float x0 = sy[b * 128 + i], x1 = sy[b * 128 + i + 64];
            float *q = p.q + ((size_t)b * d.nq + grp) * HD;
            q[i] = (x0 * cs.x - x1 * cs.y) * qscale;
            q[i + 64] = (x1 * cs.x + x0 * cs.y) * qscale;
        }
    } else {
        const bool isk = grp < d.nq + d.nkv;
        head = grp - d.nq - (isk ? 0 : d.nkv);
        // one warp per (sequence, 32-dim block): rotate (k), round to fp16, store / quantize
        for (int task = warp; task < p.B * 4; task += CW) {
            const int b = task >> 2, blk = task & 3, dd = 32 * blk + lane, pos = sh.pos[b];
            float v = sy[b * 128 + dd];
            if (isk) {
                const float2 cs = p.rope[(size_t)pos * 64 + (dd & 63)];
                const float o = sy[b * 128 + (dd ^ 64)];
                v = dd < 64 ? v * cs.x - o * cs.y : v * cs.x + o * cs.y;
            }
            const __half h = __float2half_rn(v);
            const size_t pi = ((size_t)b * d.L + l) * d.nkv + head;
            const size_t Lp = p.kv.Lp;
            if (KVT == 0) {
                if (isk) *reinterpret_cast<__half *>(p.kv.k + pi * Lp * 256 + kv_k16_off(pos, dd)) = h;
                else *reinterpret_cast<__half *>(p.kv.v + pi * Lp * 256 + kv_v16_off(dd, pos)) = h;
            } else {
                float x = __half2float(h);
                float amax = fabsf(x);
                for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, o));
                uint16_t sbits = 0;
                int q = 0;
                if (amax != 0.0f) {
                    const float dq = __fdiv_rn(amax, 127.0f);
                    sbits = __half_as_ushort(__float2half_rn(dq));
                    q = max(-127, min(127, __float2int_rn(__fdiv_rn(x, dq))));
                }
                if (isk) {
                    *reinterpret_cast<int8_t *>(p.kv.k + pi * Lp * 128 + kv_k8_off(pos, dd)) = (int8_t)q;
                    if (lane == 0) *reinterpret_cast<uint16_t *>(p.kv.ks + pi * Lp * 8 + kv_ks_off(pos, blk)) = sbits;
                } else {
                    *reinterpret_cast<int8_t *>(p.kv.v + pi * Lp * 128 + kv_v8_off(dd, pos)) = (int8_t)q;
                    if (lane == 0) *reinterpret_cast<uint16_t *>(p.kv.vs + pi * Lp * 8 + kv_vs_off(blk, pos)) = sbits;
                }
            }
        }
    }
    publish(p, c_qkvh(d, l, head));
}

// x += y on the group's 128 rows; the next projection's operand gain * x
// (planes + sub-block sums) and the group's sum of x^2 per column.
__device__ void resid_epilogue(const StepParams &p, const Dims &d, int grp, float *sy, const float *gain,
                               __half *nhi, __half *nlo, __half *nsx, float *rms_out, float *capture) {
    const int t = threadIdx.x;
    for (int task = t; task < p.B * 128; task += CTHREADS) {
        const int b = task >> 7, i = task & 127;
        float *xp = p.x + (size_t)b * d.H + grp * 128 + i;
        const float xn = __ldcg(xp) + sy[b * 128 + i];
        *xp = xn;
        if (capture) capture[(size_t)b * d.H + grp * 128 + i] = xn;
        sy[b * 128 + i] = xn;
    }
    cbar();
    if (t < p.B * 16) {   // (column, chunk of 8 rows): 16 consecutive lanes per column
        const int b = t >> 4, ch = t & 15;
        const int r0 = grp * 128 + ch * 8;
        float yy[8], part = 0.0f, sq = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; e++) {
            const float xv = sy[b * 128 + ch * 8 + e];
            sq = fmaf(xv, xv, sq);
            yy[e] = xv * gain[r0 + e];
            part += yy[e];
        }
        store_act8(nhi, nlo, act_chunk(r0 >> 8, b, (r0 & 255) >> 3, p.B), yy);
        const uint32_t m = __activemask();
        part += __shfl_xor_sync(m, part, 1);
        part += __shfl_xor_sync(m, part, 2);
        if ((ch & 3) == 0) store_sum(nsx, r0 >> 8, b, (r0 & 255) >> 5, p.B, part);
        sq += __shfl_xor_sync(m, sq, 1);
        sq += __shfl_xor_sync(m, sq, 2);
        sq += __shfl_xor_sync(m, sq, 4);
        sq += __shfl_xor_sync(m, sq, 8);
        if (ch == 0) rms_out[grp * MAX_B + b] = sq;
    }
}

// tile rows 0-7 gate, 8-15 up of ffn rows 8*rt..8*rt+7: a = silu(gate) * up
template <int NT>
__device__ void swiglu_epilogue(const StepParams &p, const StepShared &sh, int grp, const float (&y)[NT][2],
                                float *sy) {
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31, g = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int nt = 0; nt < NT; nt++) {
        const int b = 4 * nt + tig;
        if (b < p.B) sy[b * 64 + warp * 8 + g] = silu_f(y[nt][0] * sh.r[b]) * (y[nt][1] * sh.r[b]);
    }
    cbar();
    if (t < p.B * 8) {
        const int b = t >> 3, ch = t & 7;
        const int f = grp * 64 + ch * 8;
        float yy[8], part = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; e++) {
            yy[e] = sy[b * 64 + ch * 8 + e];
            part += yy[e];
        }
        store_act8(p.a16, p.a16lo, act_chunk(f >> 8, b, (f & 255) >> 3, p.B), yy);
        const uint32_t m = __activemask();
        part += __shfl_xor_sync(m, part, 1);
        part += __shfl_xor_sync(m, part, 2);
        if ((ch & 3) == 0) store_sum(p.asx, f >> 8, b, (f & 255) >> 5, p.B, part);
    }
}

// logits + the group's argmax per column; the CTA completing the last group
// reduces all groups to the ids
template <int NT>
__device__ void lm_epilogue(const StepParams &p, const Dims &d, StepShared &sh, int grp, const float (&y)[NT][2],
                            float *scr) {
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31, g = lane >> 2, tig = lane & 3;
    float *sv = scr;                                   // [8 warps][8 cols]
    int *si = reinterpret_cast<int *>(scr + CW * 8);   // [8][8]
    const int rt = grp * GT + warp;
#pragma unroll
    for (int nt = 0; nt < NT; nt++) {
        const int b = 4 * nt + tig;
        const int r0 = rt * 16 + g, r1 = r0 + 8;
        const float y0 = y[nt][0] * (b < p.B ? sh.r[b] : 0.0f), y1 = y[nt][1] * (b < p.B ? sh.r[b] : 0.0f);
        const bool v0 = rt < d.nrt_lm && r0 < d.V, v1 = rt < d.nrt_lm && r1 < d.V;
        if (p.logits && b < p.B) {
            if (v0) p.logits[(size_t)b * d.V + r0] = y0;
            if (v1) p.logits[(size_t)b * d.V + r1] = y1;
        }
        float bv = v0 ? y0 : -INFINITY;
        int bi = v0 ? r0 : 0x7FFFFFFF;
        if (v1 && y1 > bv) { bv = y1; bi = r1; }
        for (int o = 4; o < 32; o <<= 1) {
            const float ov = __shfl_xor_sync(FULL, bv, o);
            const int oi = __shfl_xor_sync(FULL, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (g == 0) { sv[warp * 8 + b] = bv; si[warp * 8 + b] = bi; }
    }
    cbar();
    if (t < p.B) {
        float bv = -INFINITY;
        int bi = 0x7FFFFFFF;
        for (int w = 0; w < CW; w++) {   // increasing rows
            const float v = sv[w * 8 + t];
            const int i = si[w * 8 + t];
            if (v > bv || (v == bv && i < bi)) { bv = v; bi = i; }
        }
        p.amax_val[grp * MAX_B + t] = bv;
        p.amax_idx[grp * MAX_B + t] = bi;
    }
    __threadfence();
    cbar();
    if (t == 0) {
        const int old = atomicAdd(p.cnt + d.c_lm, 1);
        sh.last = old == d.g_lm - 1;
        if (sh.last) __threadfence();
    }
    cbar();
    if (!sh.last) return;
    if (warp < p.B) {   // one warp per column over all groups (fixed order)
        const int b = warp;
        float bv = -INFINITY;
        int bi = 0x7FFFFFFF;
        for (int i = lane; i < d.g_lm; i += 32) {
            const float v = __ldcg(p.amax_val + i * MAX_B + b);
            const int ix = __ldcg(p.amax_idx + i * MAX_B + b);
            if (v > bv || (v == bv && ix < bi)) { bv = v; bi = ix; }
        }
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(FULL, bv, o);
            const int oi = __shfl_xor_sync(FULL, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        if (lane == 0) p.ids[b] = bi == 0x7FFFFFFF ? 0 : bi;
    }
}

template <int NT, int KVT>
__device__ void finish_group(const StepParams &p, const Dims &d, StepShared &sh, const Phase &f, int grp,
                             const float (&y)[NT][2], float *scr) {
    const int l = f.layer;
    switch (f.kind) {
        case PK_QKV:
            to_smem<NT>(p, scr, y, true, sh);
            cbar();
            qkv_epilogue<KVT>(p, d, sh, l, grp, scr);
            break;
        case PK_O:
            to_smem<NT>(p, scr, y, false, sh);
            cbar();
            resid_epilogue(p, d, grp, scr, p.layers[l].ffn_norm, p.g16, p.g16lo, p.gsx, p.rms_ffn, nullptr);
            publish(p, c_o(d, l));
            break;
        case PK_GU:
            swiglu_epilogue<NT>(p, sh, grp, y, scr);
            publish(p, c_gu(d, l));
            break;
        case PK_DOWN: {
            to_smem<NT>(p, scr, y, false, sh);
            cbar();
            const float *gain = l + 1 < d.L ? p.layers[l + 1].attn_norm : p.final_norm;
            float *cap = p.capture ? p.capture + (size_t)(l + 1) * p.B * d.H : nullptr;
            resid_epilogue(p, d, grp, scr, gain, p.u16, p.u16lo, p.usx, p.rms_attn, cap);
            publish(p, c_down(d, l));
            break;
        }
        default:
            lm_epilogue<NT>(p, d, sh, grp, y, scr);
            break;
    }
    cbar();   // the scratch is free again
}

template <int NT, int KVT>
__device__ void gemm_phase(const StepParams &p, const Dims &d, StepShared &sh, const Phase &f, int ph,
                           const Ring &ring, uint32_t &it, const StageLayout &lay, float *scr) {
    const int G = f.G, cta = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, tig = lane & 3;
    const int lo = range_lo(f.U, G, cta), hi = range_lo(f.U, G, cta + 1);
    if (lo >= hi) return;
    trace(p, ph, 0);
    const float *rms = f.kind == PK_QKV || f.kind == PK_LM ? p.rms_attn : (f.kind == PK_GU ? p.rms_ffn : nullptr);
    gate_and_norm(p, sh, f.gate, f.target, rms, d.H);
    trace(p, ph, 1);
    const uint32_t act_off = ((g & 1) ? lay.lo : lay.hi) + (uint32_t)(g >> 1) * 512u + (uint32_t)tig * 128u;
    const uint32_t swz = (uint32_t)tig | ((uint32_t)((g >> 1) & 1) << 2);
    const uint32_t sum_off = (g & 1) ? lay.zero + (uint32_t)tig * 8u
                                     : lay.sums + (uint32_t)(g >> 1) * 32u + (uint32_t)tig * 8u;
    int x = lo;
    while (x < hi) {
        const int grp = x / f.nsb;
        const int end = min(hi, (grp + 1) * f.nsb), n = end - x;
        const int rt = grp * GT + warp;
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
#pragma unroll
            for (int i = 0; i < 4; i++) acc[nt][i] = 0.0f;
        for (int i = 0; i < n; i++, it++) {
            wait_item(p, ring, it, sh);
            if (x == lo && i == 0) trace(p, ph, 2);
            if (rt < f.nrt) stage_mma<NT>(ring.slot(it), warp, lane, act_off, sum_off, swz, acc);
            release_item(ring, it, 1);
        }
        trace(p, ph, 3);
        float y[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
            y[nt][0] = acc[nt][0] + acc[nt][1] * LO_UNSCALE;
            y[nt][1] = acc[nt][2] + acc[nt][3] * LO_UNSCALE;
        }
        const int first = owner_of(f.U, G, grp * f.nsb), last = owner_of(f.U, G, (grp + 1) * f.nsb - 1);
        if (first != last) {
            const int npieces = f.U >= G ? last - first + 1 : f.nsb;
            float *mine = p.gpart + (size_t)(grp + cta) * p.B * 128;
#pragma unroll
            for (int nt = 0; nt < NT; nt++) {
                const int b = 4 * nt + tig;
                if (b < p.B)
#pragma unroll
                    for (int r = 0; r < 2; r++) mine[b * 128 + warp * 16 + g + 8 * r] = y[nt][r];
            }
            if (!piece_arrive(p, sh, f.pc + grp, npieces)) { x = end; continue; }
#pragma unroll
            for (int nt = 0; nt < NT; nt++) y[nt][0] = y[nt][1] = 0.0f;
            for (int c0 = first; c0 <= last; c0 += 4) {   // four pieces' loads in flight, summed in order
                float v[4][NT][2];
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    const int c = c0 + j;
                    const bool live = c <= last && range_lo(f.U, G, c) < range_lo(f.U, G, c + 1);
                    const float *pc = p.gpart + (size_t)(grp + c) * p.B * 128;
#pragma unroll
                    for (int nt = 0; nt < NT; nt++) {
                        const int b = 4 * nt + tig;
#pragma unroll
                        for (int r = 0; r < 2; r++)
                            v[j][nt][r] = live && b < p.B ? __ldcg(pc + b * 128 + warp * 16 + g + 8 * r) : 0.0f;
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; j++)
#pragma unroll
                    for (int nt = 0; nt < NT; nt++)
#pragma unroll
                        for (int r = 0; r < 2; r++) y[nt][r] += v[j][nt][r];
            }
        }
        finish_group<NT, KVT>(p, d, sh, f, grp, y, scr);
        x = end;
    }
    trace(p, ph, 4);
}

// normalised attention output of (b, g) -> the O projection's act planes
__device__ void att_finish(const StepParams &p, const Dims &d, int l, int b, int g, float *satt) {
    const int t = threadIdx.x;
    // satt: [4 heads][HD + 4]: (M, L, -, -, O[128])
    for (int i = t; i < GROUP * HD; i += CTHREADS) {
        const int h = i >> 7, dd = i & 127;
        satt[h * (HD + 4) + 4 + dd] = satt[h * (HD + 4) + 4 + dd] / satt[h * (HD + 4) + 1];
    }
    cbar();
    if (t < 64) {   // 512 outputs = 64 chunks of 8 (elements 512g .. 512g+511)
        const int h = t >> 4, c8 = t & 15;
        float yy[8], part = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; e++) {
            yy[e] = satt[h * (HD + 4) + 4 + 8 * c8 + e];
            part += yy[e];
        }
        const int e0 = 512 * g + 128 * h + 8 * c8;
        store_act8(p.o16, p.o16lo, act_chunk(e0 >> 8, b, (e0 & 255) >> 3, p.B), yy);
        part += __shfl_xor_sync(FULL, part, 1);
        part += __shfl_xor_sync(FULL, part, 2);
        if ((c8 & 3) == 0) store_sum(p.osx, e0 >> 8, b, (e0 & 255) >> 5, p.B, part);
    }
    publish(p, c_att(d, l));
    cbar();
}

template <int KVT>
__device__ void att_phase(const StepParams &p, const Dims &d, StepShared &sh, const Phase &f, int ph,
                          const Ring &ring, uint32_t &it, float *scr) {
    const int G = f.G, cta = blockIdx.x;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31, gid = lane >> 2, tig = lane & 3;
    const int lo = cta < G ? range_lo(f.U, G, cta) : 0, hi = cta < G ? range_lo(f.U, G, cta + 1) : 0;
    if (lo < hi) trace(p, ph, 0);
    const int pair = warp >> 1, hh = warp & 1;
    float *pm = scr;                      // [4 pairs][4 heads]
    float *pl = scr + 16;                 // [4][4]
    float *po = scr + 32;                 // [4 pairs][4 heads][128]
    float *satt = scr + 32 + 4 * 4 * HD;  // [4 heads][HD + 4]
    int x = lo;
    while (x < hi) {
        int b, g, u0, nu;
        att_item(sh, d.nkv, p.B, x, b, g, u0, nu);
        const int end = min(hi, x + (nu - u0)), n = end - x;
        const int ntok = sh.pos[b] + 1;
        gate_and_norm(p, sh, c_qkvh(d, f.layer, g), QKV_PER_HEAD, nullptr, 0);
        if (x == lo) trace(p, ph, 1);
        uint32_t qa[8][4];
        {
            const float *qr = p.q + ((size_t)b * d.nq + GROUP * g + (gid < GROUP ? gid : 0)) * HD;
#pragma unroll
            for (int s8 = 0; s8 < 8; s8++) {
                float v[4];
#pragma unroll
                for (int e = 0; e < 4; e++) v[e] = gid < GROUP ? __ldcg(qr + 16 * s8 + 4 * tig + e) : 0.0f;
                const __half2 h01 = __floats2half2_rn(v[0], v[1]), h23 = __floats2half2_rn(v[2], v[3]);
                const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
                qa[s8][0] = h2_as_u32(h01);
                qa[s8][1] = h2_as_u32(__floats2half2_rn(v[0] - f01.x, v[1] - f01.y));
                qa[s8][2] = h2_as_u32(h23);
                qa[s8][3] = h2_as_u32(__floats2half2_rn(v[2] - f23.x, v[3] - f23.y));
            }
        }
        float m_run = -INFINITY, l_run = 0.0f, oacc[8][4];
#pragma unroll
        for (int dn = 0; dn < 8; dn++)
#pragma unroll
            for (int i = 0; i < 4; i++) oacc[dn][i] = 0.0f;
        // pair q takes the items whose absolute index is q mod P (P | S, P <= 4)
        const int P = ring.S % 4 == 0 ? 4 : (ring.S % 3 == 0 ? 3 : (ring.S % 2 == 0 ? 2 : 1));
        const int i0 = pair < P ? (int)((pair + P - it % (uint32_t)P) % (uint32_t)P) : n;
        for (int i = i0; i < n; i += P) {
            const uint32_t iti = it + i;
            wait_item(p, ring, iti, sh);
            if (x == lo && i == 0) trace(p, ph, 2);
            const int u = u0 + i;
            att_unit<KVT>(ring.slot(iti), min(KU, ntok - KU * u), hh, qa, m_run, l_run, oacc);
            release_item(ring, iti, 4);
        }
        it += n;
        cbar();
        trace(p, ph, 3);
        // merge the pairs
        float l_tot = l_run;
        l_tot += __shfl_xor_sync(FULL, l_tot, 1);
        l_tot += __shfl_xor_sync(FULL, l_tot, 2);
        if (gid < GROUP) {
            if (hh == 0 && tig == 0) { pm[pair * 4 + gid] = m_run; pl[pair * 4 + gid] = l_tot; }
#pragma unroll
            for (int dn = 0; dn < 8; dn++)
#pragma unroll
                for (int e = 0; e < 2; e++)
                    po[(pair * 4 + gid) * HD + 64 * hh + 8 * dn + 2 * tig + e] = oacc[dn][e] + oacc[dn][2 + e];
        }
        cbar();
        {
            const int h = t >> 6, d0 = (t & 63) * 2;
            float M = -INFINITY;
            for (int q = 0; q < 4; q++) M = fmaxf(M, pm[q * 4 + h]);
            float L = 0.0f, O0 = 0.0f, O1 = 0.0f;
            for (int q = 0; q < 4; q++) {
                const float mq = pm[q * 4 + h];
                const float fq = mq == -INFINITY ? 0.0f : expf(mq - M);
                L += fq * pl[q * 4 + h];
                O0 += fq * po[(q * 4 + h) * HD + d0];
                O1 += fq * po[(q * 4 + h) * HD + d0 + 1];
            }
            if ((t & 63) == 0) { satt[h * (HD + 4)] = M; satt[h * (HD + 4) + 1] = L; }
            satt[h * (HD + 4) + 4 + d0] = O0;
            satt[h * (HD + 4) + 4 + d0 + 1] = O1;
        }
        cbar();
        // pieces of (b, g) across CTAs
        const int bg = b * d.nkv + g;
        const int ibeg = d.nkv * sh.units[b] + g * nu;   // first item of (b, g)
        const int first = owner_of(f.U, G, ibeg), last = owner_of(f.U, G, ibeg + nu - 1);
        if (first != last) {
            const int npieces = f.U >= G ? last - first + 1 : nu;
            float *mine = p.apart + (size_t)(bg + cta) * GROUP * (HD + 4);
            for (int i = t; i < GROUP * (HD + 4); i += CTHREADS) mine[i] = satt[i];
            if (!piece_arrive(p, sh, f.pc + bg, npieces)) { x = end; continue; }
            // merge all pieces in CTA order: loads of up to 8 pieces in flight
            const int h = t >> 6, d0 = (t & 63) * 2;
            float M = -INFINITY, L = 0.0f, O0 = 0.0f, O1 = 0.0f;
            for (int c0 = first; c0 <= last; c0 += 8) {
                float mc[8], lc[8], oa[8], ob[8];
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    const int c = c0 + j;
                    mc[j] = -INFINITY;
                    lc[j] = oa[j] = ob[j] = 0.0f;
                    if (c <= last && range_lo(f.U, G, c) < range_lo(f.U, G, c + 1)) {
                        const float *pp = p.apart + ((size_t)(bg + c) * GROUP + h) * (HD + 4);
                        mc[j] = __ldcg(pp);
                        lc[j] = __ldcg(pp + 1);
                        oa[j] = __ldcg(pp + 4 + d0);
                        ob[j] = __ldcg(pp + 4 + d0 + 1);
                    }
                }
#pragma unroll
                for (int j = 0; j < 8; j++) {   // online rescaling, pieces in CTA order
                    if (mc[j] == -INFINITY) continue;
                    const float Mn = fmaxf(M, mc[j]);
                    const float a = M == -INFINITY ? 0.0f : expf(M - Mn), bsc = expf(mc[j] - Mn);
                    L = L * a + lc[j] * bsc;
                    O0 = O0 * a + oa[j] * bsc;
                    O1 = O1 * a + ob[j] * bsc;
                    M = Mn;
                }
            }
            cbar();   // everyone has read satt's old contents
            if ((t & 63) == 0) { satt[h * (HD + 4)] = M; satt[h * (HD + 4) + 1] = L; }
            satt[h * (HD + 4) + 4 + d0] = O0;
            satt[h * (HD + 4) + 4 + d0 + 1] = O1;
            cbar();
        }
        att_finish(p, d, f.layer, b, g, satt);
        x = end;
    }
    if (lo < hi) trace(p, ph, 4);
}

// ----------------------------------------------------------------- kernel
template <int NT, int KVT>
__global__ __maxnreg__(112) void step_kernel(const StepParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ StepShared sh;
    __shared__ __align__(16) float scr[32 + 4 * 4 * HD + GROUP * (HD + 4)];
    if (*reinterpret_cast<volatile const int *>(p.step_ok) == 0) return;   // inputs rejected by the prep kernel
    const Dims d = make_dims(p.n_layers, p.hidden, p.ffn, p.vocab, p.n_q, p.n_kv);
    const int S = p.slots;
    const StageLayout lay(4 * NT);
    Ring ring;
    ring.base = smem;
    ring.S = S;
    ring.SB = (uint32_t)p.slot_bytes;
    ring.full = reinterpret_cast<uint64_t *>(smem + (size_t)S * p.slot_bytes);
    ring.empty = ring.full + S;
    const int t = threadIdx.x;
    if (t == 0) {
        sh.abort = 0;
        sh.last = 0;
        sh.units[0] = 0;
        for (int b = 0; b < p.B; b++) {
            sh.pos[b] = p.positions[b];
            sh.units[b + 1] = sh.units[b] + (sh.pos[b] + KU) / KU;
        }
        for (int i = 0; i < S; i++) {
            mbar_init(&ring.full[i], 1);
            mbar_init(&ring.empty[i], CW);
        }
        mbar_fence_init();
    }
    // zero the batch rows B..4NT-1 of every slot's activation area and the
    // lo lanes' min-term slots (the copies never write them)
    const int BR = 4 * NT;
    for (int i = t; i < S * BR * 8; i += STEP_THREADS) {
        const int s = i / (BR * 8), r = (i / 8) % BR, w = i % 8;
        uint8_t *base = smem + (size_t)s * p.slot_bytes;
        if (r >= p.B) {
            for (int k = 0; k < 4; k++) {
                *reinterpret_cast<uint4 *>(base + lay.hi + r * 512 + (w * 4 + k) * 16) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4 *>(base + lay.lo + r * 512 + (w * 4 + k) * 16) = make_uint4(0, 0, 0, 0);
            }
            if (w < 2) *reinterpret_cast<uint4 *>(base + lay.sums + r * 32 + w * 16) = make_uint4(0, 0, 0, 0);
        }
        if (w < 2) *reinterpret_cast<uint4 *>(base + lay.zero + r * 32 + w * 16) = make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
    if (t >= CTHREADS) {
        if (t == CTHREADS) producer<KVT>(p, d, sh, smem, ring.full, ring.empty, lay);
        return;
    }
    uint32_t it = 0;
    const int NPH = n_phases(d);
    for (int ph = 0; ph < NPH; ph++) {
        const Phase f = make_phase(p, d, sh, ph);
        if (f.kind == PK_EMBED) {
            trace(p, ph, 0);
            embed_phase(p, d, sh, scr);
            trace(p, ph, 4);
        } else if (f.kind == PK_ATT) att_phase<KVT>(p, d, sh, f, ph, ring, it, scr);
        else gemm_phase<NT, KVT>(p, d, sh, f, ph, ring, it, lay, scr);
    }
}

// Prep: zero the counters, check the inputs, advance the lengths.
__global__ void step_prep_kernel(int *cnt, int n_cnt, int *step_ok, int *abort_flag, uint32_t *status,
                                 const int32_t *tokens, const int32_t *positions, int32_t *len_dev, int B,
                                 int max_L, int vocab) {
    for (int i = threadIdx.x; i < n_cnt; i += blockDim.x) cnt[i] = 0;
    __shared__ int bad;
    if (threadIdx.x == 0) bad = 0;
    __syncthreads();
    if (threadIdx.x < B) {
        const int b = threadIdx.x, pos = positions[b], tok = tokens[b];
        if (pos < 0 || pos >= max_L || pos != len_dev[b]) { atomicOr(status, STATUS_POSITION); bad = 1; }
        if (tok < 0 || tok >= vocab) { atomicOr(status, STATUS_TOKEN); bad = 1; }
    }
    __syncthreads();
    if (threadIdx.x < B && !bad) len_dev[threadIdx.x] = positions[threadIdx.x] + 1;
    if (threadIdx.x == 0) {
        *step_ok = bad ? 0 : 1;
        *abort_flag = 0;
    }
}

template <int NT, int KVT>
cudaError_t launch_step_t(const StepParams &p, int grid, cudaStream_t stream, size_t smem) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(STEP_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, step_kernel<NT, KVT>, p);
}

template <int NT, int KVT>
cudaError_t setup_t(size_t smem, int *per_sm) {
    cudaError_t e = cudaFuncSetAttribute(step_kernel<NT, KVT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // all of the unified L1/shared storage as shared memory: two CTAs per SM
    e = cudaFuncSetAttribute(step_kernel<NT, KVT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, step_kernel<NT, KVT>, STEP_THREADS, smem);
}

}  // namespace

int step_counter_count(int n_layers, int hidden, int ffn, int vocab, int n_q, int n_kv) {
    return make_dims(n_layers, hidden, ffn, vocab, n_q, n_kv).n_cnt;
}
int step_lm_groups(int vocab) { return n_groups((vocab + 15) / 16); }
size_t step_gpart_floats(int hidden, int ffn, int vocab, int n_q, int n_kv, int B, int grid) {
    const Dims d = make_dims(1, hidden, ffn, vocab, n_q, n_kv);
    int gmax = d.g_qkv;
    gmax = gmax > d.g_o ? gmax : d.g_o;
    gmax = gmax > d.g_gu ? gmax : d.g_gu;
    gmax = gmax > d.g_down ? gmax : d.g_down;
    gmax = gmax > d.g_lm ? gmax : d.g_lm;
    return (size_t)(gmax + grid) * B * 128;
}
size_t step_apart_floats(int n_kv, int B, int grid) { return (size_t)(B * n_kv + grid) * GROUP * (HD + 4); }
int step_slot_bytes(int B) { return (int)StageLayout(B <= 4 ? 4 : 8).bytes; }
size_t step_smem_bytes(int B, int slots) { return (size_t)slots * step_slot_bytes(B) + (size_t)slots * 16; }

cudaError_t step_setup(int B, int kv_dtype, int slots, int *per_sm) {
    const size_t smem = step_smem_bytes(B, slots);
    if (B <= 4) return kv_dtype ? setup_t<1, 1>(smem, per_sm) : setup_t<1, 0>(smem, per_sm);
    return kv_dtype ? setup_t<2, 1>(smem, per_sm) : setup_t<2, 0>(smem, per_sm);
}

cudaError_t launch_step(const StepParams &p, int grid, int32_t *len_dev, cudaStream_t stream) {
    if (p.B < 1 || p.B > STEP_MAX_B) return cudaErrorInvalidValue;
    step_prep_kernel<<<1, 256, 0, stream>>>(p.cnt, p.n_cnt, const_cast<int *>(p.step_ok), p.abort_flag, p.status,
                                            p.tokens, p.positions, len_dev, p.B, p.max_L, p.vocab);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t smem = step_smem_bytes(p.B, p.slots);
    if (p.B <= 4)
        return p.kv.kv_dtype ? launch_step_t<1, 1>(p, grid, stream, smem) : launch_step_t<1, 0>(p, grid, stream, smem);
    return p.kv.kv_dtype ? launch_step_t<2, 1>(p, grid, stream, smem) : launch_step_t<2, 0>(p, grid, stream, smem);
}

}  // namespace zdec
