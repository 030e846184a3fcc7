// et_gemm.cuh -- persistent, warp-specialised tile-GEMM pipeline:
//   D[128 weight rows, n token rows] = sum_k W[a_row.., k] * Act[b_row.., k]
// with the weight tile on the UMMA M side ("swap-AB": decode-sized token
// counts sit on N, which may be as small as 16 and as large as 256).
//
// Each role runs its own loop over the CTA's task sequence and meets the
// others only through mbarriers -- there is no CTA-wide barrier inside a loop:
//   warp 0 lane 0   TMA producer: reserves ring space for one k-block fill,
//                   posts its byte count, loads the weight tile(s) and the
//                   activation rows; a task with a dependency loads the
//                   weight tiles of the fills that fit *before* it waits on
//                   the event, so the weight stream is already in flight
//                   when the dependency resolves;
//   warp 1 lane 0   MMA issuer: per task, waits for free TMEM accumulator
//                   slots, issues tcgen05.mma per full fill, frees each fill
//                   with tcgen05.commit, commits the accumulator slots;
//   warps 2..9      workers: the epilogue (tcgen05.ld from TMEM, stores,
//                   event releases) and every non-GEMM task; they sync among
//                   themselves with named barrier 1.  Warp w may only read TMEM
//                   lanes 32*(w%4) ..; warps 2..5 take the even 16-column chunks
//                   of an accumulator, warps 6..9 the odd ones, so each lane
//                   quadrant is read by one warp of each half.
//
// The stage ring is byte-granular: a fill takes exactly the bytes of its
// k-block (weights 16 or 32 KB, plus n * 128 bytes of activation rows), so a
// decode-sized task keeps many more weight bytes in flight than a wide one.
// Producer and MMA issuer place fills with the same deterministic rule; only
// the producer waits for space, releasing older fills in order.
//
// TMEM holds two accumulator slots of 256 columns.  A task takes one slot
// (gate and up side by side when n <= 128) or both (gate/up with n > 128), so
// the MMA of the next task overlaps the epilogue of the last one whenever the
// accumulators fit.
#pragma once

#include "et_device.cuh"

namespace et {

constexpr int kTaskRing = 4;       // dynamic-queue tasks handed from producer to consumers
constexpr int kWorkers = 256;      // warps 2..9
constexpr int kWorkerBar = 1;      // named barrier id of the worker group
constexpr int kSlots = 16;         // ring fills in flight at most (one barrier pair each)
constexpr int kAccSlotCols = 256;  // TMEM columns per accumulator slot

// One task as handed through the smem ring (dynamic schedules).
struct TaskMsg {
    int32_t type, a, b, c;  // type | (split << 8), then task-specific indices
    int32_t e, row0, rows, n;
    uint32_t aux;           // MoE gate/up tile of a one-router-tile batch: its tokens (bit t)
};

// Per-CTA control block, after the stage ring and the SIMT scratch in smem.
struct Ctl {
    uint64_t full[kSlots];
    uint64_t empty[kSlots];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t tq_full[kTaskRing];
    uint64_t tq_empty[kTaskRing];
    uint64_t drain;
    uint64_t sbar;                // worker staging copies (bulk async)
    TaskMsg tq[kTaskRing];
    uint32_t unit_end[kSlots];    // producer: ring end position of each fill in flight
    uint32_t tmem_base;
    int32_t issued;    // fills posted by the producer (for the unwind)
    int32_t consumed;  // fills consumed by the MMA issuer
    int32_t flag;      // worker broadcast
    int32_t wflag[2];  // worker_wait decisions, double buffered
    int32_t ring_ret;  // ring leases the workers have returned
    int32_t scratch[16];
    uint32_t post_ns[kSlots];  // trace: low word of %globaltimer when each fill was posted
};

// The byte ring of stage fills.
struct Ring {
    uint8_t* base;
    uint32_t bytes;
};

struct GemmTask {
    const CUtensorMap* a0;   // weight map, box 64 x 128
    const CUtensorMap* a1;   // second weight map (gate/up) or nullptr
    const CUtensorMap* b;    // activation map, box 64 x 16
    const CUtensorMap* b64;  // the same activations, box 64 x 64
    int a_row;               // first weight row
    int b_row;               // first activation row
    int kb0, nkb;            // k-blocks [kb0, kb0 + nkb), 64 elements each
    int n;                   // UMMA N: multiple of 16, <= 256
    const int* dep;          // wait *dep >= dep_target before activation loads
    int dep_target;
    int dep_where;
    int a1_off = 0;          // row offset of the second weight tile (gate/up: 0, same rows of
                             // another matrix; a 256-row down tile: 128, the next rows)
};

// One k-block: [A0 16K][A1 16K if gate/up][B n*128].  A fill packs several
// consecutive k-blocks -- four when one is at most 24 KB (a narrow down tile),
// two up to 48 KB -- so each weight row is requested 256..512 contiguous bytes
// at a time and fewer fills are tracked.  Measured on GB300 against one
// k-block per fill: 15 % less time for a Mixtral-shaped layer at 16..64
// tokens and 10 % at 512 (fewer, longer DRAM row accesses).
__device__ __forceinline__ uint32_t kblock_bytes(const GemmTask& t) {
    return (t.a1 ? 2u : 1u) * kABytes + static_cast<uint32_t>(t.n) * 128u;
}
__device__ __forceinline__ int kpack_of(const GemmTask& t) {
    const uint32_t b = kblock_bytes(t);
    return b <= 24576u ? 4 : (b <= 49152u ? 2 : 1);
}
__device__ __forceinline__ int fills_of(const GemmTask& t) { return ceil_div(t.nkb, kpack_of(t)); }
// First k-block (relative to kb0) and k-block count of the task's u-th fill.
// Every task walks its k-blocks in order: concurrent tiles of neighbouring
// weight rows then read the same columns at the same time, which streams DRAM
// faster than staggered starts (measured: +2.5 % over the Mixtral sweep).
__device__ __forceinline__ int fill_kb(const GemmTask& t, int u, int& nk) {
    const int kp = kpack_of(t);
    const int kb = u * kp;
    nk = min(kp, t.nkb - kb);
    return kb;
}
// Fill layout: [A0 x kp][A1 x kp][B x kp] (every tile 1024-byte aligned); a
// ragged last fill is placed with the full size.
__device__ __forceinline__ uint32_t unit_bytes(const GemmTask& t) {
    return static_cast<uint32_t>(kpack_of(t)) * kblock_bytes(t);
}

// TMEM accumulator slots a task takes: gate/up needs 2n columns.
__host__ __device__ __forceinline__ uint32_t acc_slots(bool two, int n) {
    return (two ? 2 * n : n) > kAccSlotCols ? 2u : 1u;
}

// Ring placement shared by producer and MMA issuer: a fill that would run
// past the end starts again at offset 0.  Positions are monotonic; the
// address is base + position % bytes.
__device__ __forceinline__ uint32_t ring_place(uint32_t& head, uint32_t sb, uint32_t rb) {
    const uint32_t off = head % rb;
    if (off + sb > rb) head += rb - off;
    const uint32_t start = head;
    head += sb;
    return start;
}

// ------------------------------------------------------------------ trace

// Optional per-task record (see et_opts.trace): {type | role << 8, a, b, cta,
// t_begin, t_end}.  Each CTA owns an equal share of the buffer's records and
// fills it through a shared-memory counter, so a record costs plain stores
// (no global atomic on the path being timed); records beyond a CTA's share
// are dropped, unused ones stay zero.
__device__ __forceinline__ unsigned* trace_counter() {
    __shared__ unsigned n;
    return &n;
}
__device__ __forceinline__ void trace_init() {  // thread 0, before the CTA's first barrier
    *trace_counter() = 0;
}
__device__ __forceinline__ void trace_put(uint64_t* buf, int cap, int type, int role, int a,
                                          int b, uint64_t t0, uint64_t t1) {
    if (!buf) return;
    const unsigned per = static_cast<unsigned>(cap) / gridDim.x;
    const unsigned i = atomicAdd(trace_counter(), 1u);
    if (i >= per) return;
    int4* r = reinterpret_cast<int4*>(reinterpret_cast<uint8_t*>(buf) + 32 +
                                      (static_cast<size_t>(blockIdx.x) * per + i) * 32);
    r[0] = make_int4(type | (role << 8), a, b, static_cast<int>(blockIdx.x));
    uint64_t* t = reinterpret_cast<uint64_t*>(r + 1);
    t[0] = t0;
    t[1] = t1;
}

// Records a worker task (role 1) when it leaves scope, on any path.
struct TraceOnExit {
    uint64_t* buf;
    int cap, type, a;
    uint64_t t0;
    bool on;
    __device__ __forceinline__ ~TraceOnExit() {
        if (on && buf) trace_put(buf, cap, type, 1, a, 0, t0, globaltimer_ns());
    }
};

// ------------------------------------------------------------------ producer

struct ProdState {
    uint32_t it = 0;    // fills posted
    uint32_t head = 0;  // ring position after the last placed fill
    uint32_t rel = 0;   // fills known to be released
    uint32_t tail = 0;  // ring end position of the newest released fill
    uint32_t leases = 0;  // SIMT tasks handed to the workers (each leases the ring)
};

// A SIMT task may use the ring as staging space: the producer hands it over
// (a lease) and posts no fill until the workers have returned every lease.
// Every earlier fill is already consumed when the workers start that task
// (they take tasks in order, after the epilogue of the last GEMM).
__device__ __forceinline__ bool ring_lease_wait(Ctl* ctl, const ProdState& ps, const WaitCtx& wc) {
    const volatile int32_t* ret = &ctl->ring_ret;
    if (*ret < static_cast<int32_t>(ps.leases)) {
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t it = 1; *ret < static_cast<int32_t>(ps.leases); ++it) {
            __nanosleep(it > 32 ? 256 : 32);  // (a lease lasts a whole SIMT task)
            if ((it & 15u) == 0) {
                if (aborted(wc)) return false;
                if (globaltimer_ns() - t0 > wc.timeout_ns) {
                    raise_error(wc, ET_ERR_TIMEOUT, kWhereStage);
                    return false;
                }
            }
        }
    }
    fence_proxy_async_smem();  // the workers' use of the ring precedes the next TMA writes
    return true;
}

// Wait, oldest first, for released fills until a fill of `sb` bytes at
// `start` has both a barrier slot and its bytes free.
__device__ __forceinline__ bool ring_reserve(Ctl* ctl, ProdState& ps, uint32_t start, uint32_t sb,
                                             uint32_t rb, const WaitCtx& wc) {
    while (ps.rel < ps.it && (ps.it - ps.rel >= static_cast<uint32_t>(kSlots) ||
                              start + sb > ps.tail + rb)) {
        const uint32_t slot = ps.rel % kSlots;
        if (!mbar_wait(wc, &ctl->empty[slot], (ps.rel / kSlots) & 1u, kWhereEmpty)) return false;
        ps.tail = ctl->unit_end[slot];
        ++ps.rel;
    }
    return true;
}

// Reserve and post fill `u` of task t (its byte count, its weight tiles).
__device__ __forceinline__ bool post_weights(const GemmTask& t, const Ring& R, Ctl* ctl,
                                             ProdState& ps, int u, const WaitCtx& wc,
                                             uint64_t pol_w) {
    const uint32_t sb = unit_bytes(t);
    const uint32_t start = ring_place(ps.head, sb, R.bytes);
    if (!ring_reserve(ctl, ps, start, sb, R.bytes, wc)) return false;
    const uint32_t slot = ps.it % kSlots;
    ctl->unit_end[slot] = start + sb;
    const int kp = kpack_of(t);
    int nk;
    const int kb = fill_kb(t, u, nk);
    mbar_arrive_expect_tx(&ctl->full[slot], static_cast<uint32_t>(nk) * kblock_bytes(t));
    uint8_t* dst = R.base + start % R.bytes;
    for (int j = 0; j < nk; ++j) {
        const int kx = (t.kb0 + kb + j) * kBlockK;
        tma_load_2d(dst + j * kABytes, t.a0, &ctl->full[slot], kx, t.a_row, pol_w);
        if (t.a1)
            tma_load_2d(dst + (kp + j) * kABytes, t.a1, &ctl->full[slot], kx, t.a_row + t.a1_off,
                        pol_w);
    }
    ++ps.it;
    return true;
}

// Activation rows of fill number `f` (already posted) = fill u of task t.
__device__ __forceinline__ void load_acts(const GemmTask& t, const Ring& R, Ctl* ctl, uint32_t f,
                                          int u, uint64_t pol_b) {
    const uint32_t slot = f % kSlots;
    const uint32_t start = ctl->unit_end[slot] - unit_bytes(t);
    const int kp = kpack_of(t);
    int nk;
    const int kb = fill_kb(t, u, nk);
    const uint32_t bbytes = static_cast<uint32_t>(t.n) * 128u;
    uint8_t* bb = R.base + start % R.bytes + static_cast<uint32_t>(kp) * (t.a1 ? 2u : 1u) * kABytes;
    const int n64 = t.b64 ? t.n / kBBoxRowsWide * kBBoxRowsWide : 0;  // rows in 64-row boxes
    for (int j = 0; j < nk; ++j) {
        const int kx = (t.kb0 + kb + j) * kBlockK;
        uint8_t* bj = bb + j * bbytes;
        for (int r = 0; r < n64; r += kBBoxRowsWide)
            tma_load_2d(bj + r * 128, t.b64, &ctl->full[slot], kx, t.b_row + r, pol_b);
        for (int r = n64; r < t.n; r += kBBoxRows)
            tma_load_2d(bj + r * 128, t.b, &ctl->full[slot], kx, t.b_row + r, pol_b);
    }
}

// ------------------------------------------------------------------ producer lookahead

// A GEMM task whose fills are being posted.  Fills are posted in task order
// (every fill of a task before any fill of the next), so the MMA issuer, which
// walks tasks and fills in order, is unchanged.  While the current task waits
// on its dependency, the producer requests the weight tiles of the CTA's next
// task into ring space that is free at that moment -- it never waits for
// space on the next task's behalf, so the fills the current task needs can
// always be placed -- and a dependency wait no longer leaves the ring idle.
struct Flight {
    GemmTask t;
    uint32_t f0;    // ring fill number of the task's first fill
    int nfill;      // fills in all
    int posted;     // fills whose weight tiles are requested
    int acts;       // ... whose activation rows are requested too
    bool ready;     // the dependency is met (or there is none)
    int type, a, b; // trace: the task
    uint64_t t_pop; // trace: when the task was taken
};

__device__ __forceinline__ void flight_begin(Flight& f, const GemmTask& t, int type, int a, int b,
                                             uint64_t t_pop) {
    f.t = t;
    f.f0 = 0;
    f.nfill = fills_of(t);
    f.posted = 0;
    f.acts = 0;
    f.ready = t.dep == nullptr;
    if (!f.ready && ld_acquire(t.dep) >= t.dep_target) {
        f.ready = true;
        fence_proxy_async_global();  // rows written by other CTAs' generic stores
    }
    f.type = type;
    f.a = a;
    f.b = b;
    f.t_pop = t_pop;
}

// ring_reserve without waiting: true when a fill of `sb` bytes at `start` has
// a barrier slot and its bytes free right now (released fills are retired).
__device__ __forceinline__ bool ring_try_reserve(Ctl* ctl, ProdState& ps, uint32_t start,
                                                 uint32_t sb, uint32_t rb) {
    while (ps.rel < ps.it && (ps.it - ps.rel >= static_cast<uint32_t>(kSlots) ||
                              start + sb > ps.tail + rb)) {
        const uint32_t slot = ps.rel % kSlots;
        if (!mbar_try_wait(&ctl->empty[slot], (ps.rel / kSlots) & 1u)) return false;
        ps.tail = ctl->unit_end[slot];
        ++ps.rel;
    }
    return true;
}

// Post the next fill of f at ring position `start` (space reserved): its byte
// count and weight tiles, and its activation rows once the dependency is met.
__device__ __forceinline__ void flight_post(Flight& f, const Ring& R, Ctl* ctl, ProdState& ps,
                                            uint32_t start, uint64_t pol_w, uint64_t pol_b) {
    const GemmTask& t = f.t;
    const uint32_t slot = ps.it % kSlots;
    ctl->unit_end[slot] = start + unit_bytes(t);
    ctl->post_ns[slot] = static_cast<uint32_t>(globaltimer_ns());
    if (f.posted == 0) f.f0 = ps.it;
    const int u = f.posted, kp = kpack_of(t);
    int nk;
    const int kb = fill_kb(t, u, nk);
    mbar_arrive_expect_tx(&ctl->full[slot], static_cast<uint32_t>(nk) * kblock_bytes(t));
    uint8_t* dst = R.base + start % R.bytes;
    for (int j = 0; j < nk; ++j) {
        const int kx = (t.kb0 + kb + j) * kBlockK;
        tma_load_2d(dst + j * kABytes, t.a0, &ctl->full[slot], kx, t.a_row, pol_w);
        if (t.a1)
            tma_load_2d(dst + (kp + j) * kABytes, t.a1, &ctl->full[slot], kx, t.a_row + t.a1_off,
                        pol_w);
    }
    ++ps.it;
    ++f.posted;
    ctl->issued = static_cast<int32_t>(ps.it);
    if (f.ready) {
        load_acts(t, R, ctl, ps.it - 1, u, pol_b);
        ++f.acts;
    }
}

// Post fills of f while ring space is free now (never waits).
__device__ __forceinline__ void flight_post_nowait(Flight& f, const Ring& R, Ctl* ctl,
                                                   ProdState& ps, uint64_t pol_w, uint64_t pol_b) {
    const uint32_t sb = unit_bytes(f.t);
    while (f.posted < f.nfill) {
        uint32_t h = ps.head;
        const uint32_t start = ring_place(h, sb, R.bytes);
        if (!ring_try_reserve(ctl, ps, start, sb, R.bytes)) return;
        ps.head = h;
        flight_post(f, R, ctl, ps, start, pol_w, pol_b);
    }
}

// Wait (bounded) until f's dependency is met, then request the activation
// rows of its posted fills.  Between polls f's own weights are posted as ring
// space frees up; once every fill of f is posted, `idle()` runs instead (the
// caller looks ahead to its next task there).  Returns false on a timeout
// (recorded) or an abort.
template <class Idle>
__device__ __forceinline__ bool flight_wait(Flight& f, const Ring& R, Ctl* ctl, ProdState& ps,
                                            const WaitCtx& wc, uint64_t pol_w, uint64_t pol_b,
                                            Idle&& idle) {
    if (!f.ready) {
        const uint64_t t0 = globaltimer_ns();
        uint32_t ns = 32;
        for (;;) {
            if (f.posted < f.nfill)
                flight_post_nowait(f, R, ctl, ps, pol_w, pol_b);
            else
                idle();
            if (ld_acquire(f.t.dep) >= f.t.dep_target) break;
            if (aborted(wc)) return false;
            if (globaltimer_ns() - t0 > wc.timeout_ns) {
                raise_error(wc, ET_ERR_TIMEOUT, f.t.dep_where);
                return false;
            }
            __nanosleep(ns);
            if (ns < 256) ns <<= 1;
        }
        f.ready = true;
        fence_proxy_async_global();  // rows written by other CTAs' generic stores
    }
    for (; f.acts < f.posted; ++f.acts) load_acts(f.t, R, ctl, f.f0 + f.acts, f.acts, pol_b);
    return true;
}

// Post the remaining fills of f (its dependency met), waiting for ring space
// -- the older fills it waits for all have their activation rows requested.
__device__ __forceinline__ bool flight_finish(Flight& f, const Ring& R, Ctl* ctl, ProdState& ps,
                                              const WaitCtx& wc, uint64_t pol_w, uint64_t pol_b) {
    const uint32_t sb = unit_bytes(f.t);
    while (f.posted < f.nfill) {
        const uint32_t start = ring_place(ps.head, sb, R.bytes);
        if (!ring_reserve(ctl, ps, start, sb, R.bytes, wc)) return false;
        flight_post(f, R, ctl, ps, start, pol_w, pol_b);
    }
    return true;
}

// A static schedule's producer: the CTA's GEMM tasks in order, `next(t)`
// giving the next one (false at the end), with one task of lookahead.
template <class Next>
__device__ __forceinline__ void produce_static(Next&& next, const Ring& R, Ctl* ctl,
                                               const WaitCtx& wc, uint64_t pol_w, uint64_t pol_b) {
    ProdState ps;
    Flight fc, fn;
    bool has_next = false;
    GemmTask t;
    for (;;) {
        if (has_next) {
            fc = fn;
            has_next = false;
        } else {
            if (!next(t)) break;
            flight_begin(fc, t, 0, 0, 0, 0);
            flight_post_nowait(fc, R, ctl, ps, pol_w, pol_b);
        }
        const bool ok = flight_wait(fc, R, ctl, ps, wc, pol_w, pol_b, [&]() {
            if (!has_next && next(t)) {
                flight_begin(fn, t, 0, 0, 0, 0);
                has_next = true;
            }
            if (has_next) flight_post_nowait(fn, R, ctl, ps, pol_w, pol_b);
        });
        if (!ok || !flight_finish(fc, R, ctl, ps, wc, pol_w, pol_b)) break;
    }
}

// One task, posted whole: its fills that fit now, the dependency, then every
// remaining fill (waiting for ring space).
__device__ __forceinline__ bool produce_task(const GemmTask& t, const Ring& R, Ctl* ctl,
                                             ProdState& ps, const WaitCtx& wc, uint64_t pol_w,
                                             uint64_t pol_b) {
    if (!ring_lease_wait(ctl, ps, wc)) return false;
    Flight f;
    flight_begin(f, t, 0, 0, 0, 0);
    flight_post_nowait(f, R, ctl, ps, pol_w, pol_b);
    return flight_wait(f, R, ctl, ps, wc, pol_w, pol_b, []() {}) &&
           flight_finish(f, R, ctl, ps, wc, pol_w, pol_b);
}

// ------------------------------------------------------------------ MMA issuer

struct MmaState {
    uint32_t it = 0;    // fills consumed
    uint32_t head = 0;  // ring position (same placement as the producer)
    uint32_t acc = 0;   // accumulator slots taken
};

// A per-fill trace hook of mma_task: called as fn(u, t_posted, t_landed) (ns).
struct NoFillTrace {
    __device__ __forceinline__ void operator()(int, uint64_t, uint64_t) const {}
};

template <class FillTrace = NoFillTrace>
__device__ __forceinline__ bool mma_task(const GemmTask& t, const Ring& R, Ctl* ctl, MmaState& ms,
                                         uint32_t tmem, const WaitCtx& wc,
                                         const FillTrace& ftr = FillTrace()) {
    const uint32_t w = acc_slots(t.a1 != nullptr, t.n);
    for (uint32_t i = 0; i < w; ++i) {
        const uint32_t s = ms.acc + i;
        if (!mbar_wait(wc, &ctl->acc_empty[s & 1u], ((s >> 1) & 1u) ^ 1u, kWhereAcc)) return false;
    }
    tc_fence_after();
    const uint32_t acc0 = tmem + (ms.acc & 1u) * kAccSlotCols;
    const uint32_t acc1 =
        w == 2 ? tmem + ((ms.acc + 1) & 1u) * kAccSlotCols : acc0 + kAccSlotCols / 2;
    const uint32_t sb = unit_bytes(t);
    const int kp = kpack_of(t), nfill = fills_of(t);
    const uint32_t bbytes = static_cast<uint32_t>(t.n) * 128u;
    const uint32_t b_off = static_cast<uint32_t>(kp) * (t.a1 ? 2u : 1u) * kABytes;
    const uint32_t idesc = idesc_bf16_m128(t.n);
    for (int u = 0; u < nfill; ++u) {
        const uint32_t start = ring_place(ms.head, sb, R.bytes);
        const uint32_t slot = ms.it % kSlots;
        if (!mbar_wait(wc, &ctl->full[slot], (ms.it / kSlots) & 1u, kWhereFull)) return false;
        {
            const uint64_t now = globaltimer_ns();
            uint64_t tp = (now & ~0xffffffffull) | ctl->post_ns[slot];
            if (tp > now) tp -= 1ull << 32;
            ftr(u, tp, now);
        }
        ms.it += 1;
        ctl->consumed = static_cast<int32_t>(ms.it);
        tc_fence_after();
        const uint32_t base = smem_u32(R.base + start % R.bytes);
        int nk;
        (void)fill_kb(t, u, nk);
        for (int j = 0; j < nk; ++j) {
            const uint32_t a_s = base + j * kABytes;
            const uint32_t a1_s = base + (kp + j) * kABytes;
            const uint32_t b_s = base + b_off + j * bbytes;
#pragma unroll
            for (int kk = 0; kk < kBlockK / 16; ++kk) {
                const uint32_t accumulate = (u > 0 || j > 0 || kk > 0) ? 1u : 0u;
                const uint64_t bd = sdesc_sw128(b_s + kk * 32);
                tc_mma_bf16(acc0, sdesc_sw128(a_s + kk * 32), bd, idesc, accumulate);
                if (t.a1) tc_mma_bf16(acc1, sdesc_sw128(a1_s + kk * 32), bd, idesc, accumulate);
            }
        }
        tc_commit(&ctl->empty[slot]);
    }
    for (uint32_t i = 0; i < w; ++i) tc_commit(&ctl->acc_full[(ms.acc + i) & 1u]);
    ms.acc += w;
    return true;
}

// ------------------------------------------------------------------ workers

__device__ __forceinline__ void worker_sync() { named_bar_sync(kWorkerBar, kWorkers); }

// A bounded mbarrier wait taken by the whole worker group: one worker thread
// waits, the decision is broadcast, so all worker warps always take the
// same path (a named barrier cannot be bounded, so they must never diverge).
// `seq` is the caller's running count of worker_wait calls.
__device__ __forceinline__ bool worker_wait(Ctl* ctl, uint64_t* bar, uint32_t parity,
                                            const WaitCtx& wc, int where, uint32_t& seq) {
    const int slot = seq & 1;
    ++seq;
    if (threadIdx.x == kEpiWarp0 * 32) ctl->wflag[slot] = mbar_wait(wc, bar, parity, where) ? 1 : 0;
    worker_sync();
    return ctl->wflag[slot] != 0;
}

// The workers' view of the accumulator slots.
struct EpiState {
    uint32_t acc = 0;   // accumulator slots consumed
    uint32_t seq = 0;   // worker_wait calls
};

// Wait for the accumulator slot(s) of the workers' next GEMM task; returns
// the TMEM address (lane 0) of the first and the second accumulator.
__device__ __forceinline__ bool epi_acquire(Ctl* ctl, EpiState& es, bool two, int n, uint32_t tmem,
                                            const WaitCtx& wc, uint32_t& acc0, uint32_t& acc1) {
    const uint32_t w = acc_slots(two, n);
    for (uint32_t i = 0; i < w; ++i) {
        const uint32_t s = es.acc + i;
        if (!worker_wait(ctl, &ctl->acc_full[s & 1u], (s >> 1) & 1u, wc, kWhereAcc, es.seq))
            return false;
    }
    tc_fence_after();
    acc0 = tmem + (es.acc & 1u) * kAccSlotCols;
    acc1 = w == 2 ? tmem + ((es.acc + 1) & 1u) * kAccSlotCols : acc0 + kAccSlotCols / 2;
    return true;
}

// The worker warp is done reading the accumulator slot(s) of its task.
__device__ __forceinline__ void epi_release(Ctl* ctl, EpiState& es, bool two, int n) {
    const uint32_t w = acc_slots(two, n);
    tc_fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0)
        for (uint32_t i = 0; i < w; ++i) mbar_arrive(&ctl->acc_empty[(es.acc + i) & 1u]);
    es.acc += w;
}

// Bulk (async-proxy) staging by the workers: worker thread 0 posts `bytes`
// on the staging barrier and issues the copies; all workers then wait.
// `sphase` is the workers' running count of staging rounds.
__device__ __forceinline__ bool staging_wait(Ctl* ctl, uint32_t& sphase, const WaitCtx& wc,
                                             uint32_t& seq) {
    const uint32_t parity = sphase & 1u;
    const bool ok = worker_wait(ctl, &ctl->sbar, parity, wc, kWhereStage, seq);
    ++sphase;
    // the phase has completed: every worker observes it itself, which makes
    // the async-proxy writes visible to its own reads
    if (ok) (void)mbar_try_wait(&ctl->sbar, parity);
    return ok;
}

// The workers are done with the ring after a SIMT task: return the lease.
__device__ __forceinline__ void ring_return(Ctl* ctl) {
    worker_sync();
    if (threadIdx.x == kEpiWarp0 * 32) {
        fence_proxy_async_smem();
        __threadfence_block();
        *reinterpret_cast<volatile int32_t*>(&ctl->ring_ret) = ctl->ring_ret + 1;
    }
}

// Split reduction of one row slice: Y[r, col0 .. col0+128) =
// bf16(sum over s in order 0, 1, .. of part[s][r][col]) for r in [r0, r1).
// part + s * sstride + r * ld + col addresses partial s (fp32); the worker
// group reads float4 columns with every split's load in flight at once.
template <int kMaxSplit = 16>
__device__ __forceinline__ void reduce_slice(const float* part, size_t sstride, int ld, int split,
                                             int r0, int r1, int col0, bf16* Y, int ldy) {
    const int nv = (r1 - r0) * (kTileM / 4);
    for (int v = static_cast<int>(threadIdx.x) - kEpiWarp0 * 32; v < nv; v += kWorkers) {
        const int row = r0 + v / (kTileM / 4), col = col0 + (v % (kTileM / 4)) * 4;
        const float* src = part + static_cast<size_t>(row) * ld + col;
        float4 q[kMaxSplit];
#pragma unroll
        for (int s = 0; s < kMaxSplit; ++s)
            if (s < split) q[s] = __ldcg(reinterpret_cast<const float4*>(src + s * sstride));
        float4 acc = q[0];
#pragma unroll
        for (int s = 1; s < kMaxSplit; ++s)
            if (s < split) {
                acc.x = acc.x + q[s].x;
                acc.y = acc.y + q[s].y;
                acc.z = acc.z + q[s].z;
                acc.w = acc.w + q[s].w;
            }
        __nv_bfloat162 o[2] = {__floats2bfloat162_rn(acc.x, acc.y), __floats2bfloat162_rn(acc.z, acc.w)};
        *reinterpret_cast<uint2*>(Y + static_cast<size_t>(row) * ldy + col) =
            *reinterpret_cast<const uint2*>(o);
    }
}

// reduce_slice with at most four splits' loads in flight at a time, and not
// inlined: callers inside register-tight loops pay a register save only on
// this (rare) path.  The same sum order.
static __device__ __noinline__ void reduce_slice4(const float* part, size_t sstride, int ld,
                                                  int split, int r0, int r1, int col0, bf16* Y,
                                                  int ldy) {
    const int nv = (r1 - r0) * (kTileM / 4);
    for (int v = static_cast<int>(threadIdx.x) - kEpiWarp0 * 32; v < nv; v += kWorkers) {
        const int row = r0 + v / (kTileM / 4), col = col0 + (v % (kTileM / 4)) * 4;
        const float* src = part + static_cast<size_t>(row) * ld + col;
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        for (int s0 = 0; s0 < split; s0 += 4) {
            float4 q[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (s0 + i < split) q[i] = __ldcg(reinterpret_cast<const float4*>(src + (s0 + i) * sstride));
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (s0 + i < split) {
                    if (s0 + i == 0) {
                        acc = q[0];
                    } else {
                        acc.x = acc.x + q[i].x;
                        acc.y = acc.y + q[i].y;
                        acc.z = acc.z + q[i].z;
                        acc.w = acc.w + q[i].w;
                    }
                }
        }
        __nv_bfloat162 o[2] = {__floats2bfloat162_rn(acc.x, acc.y), __floats2bfloat162_rn(acc.z, acc.w)};
        *reinterpret_cast<uint2*>(Y + static_cast<size_t>(row) * ldy + col) =
            *reinterpret_cast<const uint2*>(o);
    }
}

// ------------------------------------------------------------------ set-up / unwind

// Stage ring bytes that fit next to `scratch` bytes of SIMT scratch.
__host__ __device__ constexpr int ring_bytes_for(int scratch) {
    return (kSmemLimit - 1024 - scratch - static_cast<int>(sizeof(Ctl))) / 1024 * 1024;
}

// Dynamic smem layout: [align 1024][ring][scratch][Ctl].
__host__ __device__ constexpr int smem_bytes_for(int scratch) {
    return 1024 + ring_bytes_for(scratch) + scratch + static_cast<int>(sizeof(Ctl));
}

__device__ __forceinline__ Ctl* cta_setup(uint8_t* smem_raw, int scratch, Ring& R,
                                          uint8_t** scratch_out) {
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    R.base = base;
    R.bytes = static_cast<uint32_t>(ring_bytes_for(scratch));
    *scratch_out = base + R.bytes;
    Ctl* ctl = reinterpret_cast<Ctl*>(base + R.bytes + scratch);
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kSlots; ++i) {
            mbar_init(&ctl->full[i], 1);
            mbar_init(&ctl->empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctl->acc_full[i], 1);
            mbar_init(&ctl->acc_empty[i], kWorkers / 32);
        }
        for (int i = 0; i < kTaskRing; ++i) {
            mbar_init(&ctl->tq_full[i], 1);
            mbar_init(&ctl->tq_empty[i], 1 + kWorkers / 32);  // MMA thread + worker warps
        }
        mbar_init(&ctl->drain, 1);
        mbar_init(&ctl->sbar, 1);
        trace_init();
        ctl->issued = 0;
        ctl->consumed = 0;
        ctl->ring_ret = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&ctl->tmem_base, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    return ctl;
}

// After every role has left its loop (call with the whole CTA): if the launch
// aborted, let this CTA's own TMA copies and MMAs land (bounded, without
// raising), then release TMEM.
__device__ __forceinline__ void cta_teardown(Ctl* ctl, bool aborted_run) {
    __syncthreads();
    if (aborted_run && threadIdx.x == 32) {
        const uint64_t budget = 2000000ull;  // 2 ms per wait
        for (uint32_t c = static_cast<uint32_t>(ctl->consumed);
             c < static_cast<uint32_t>(ctl->issued); ++c)
            mbar_drain(&ctl->full[c % kSlots], (c / kSlots) & 1u, budget);
        tc_commit(&ctl->drain);
        mbar_drain(&ctl->drain, 0, budget);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if ((threadIdx.x >> 5) == 1) tmem_dealloc(ctl->tmem_base, kTmemCols);
}

}  // namespace et
