// et_gemm.cuh -- persistent, warp-specialised tile-GEMM pipeline:
//   D[128 weight rows, n token rows] = sum_k W[a_row.., k] * Act[b_row.., k]
// with the weight tile on the UMMA M side ("swap-AB": decode-sized token
// counts sit on N, which may be as small as 16).
//
// Each role runs its own loop over the CTA's task sequence and meets the
// others only through mbarriers -- there is no CTA-wide barrier inside a loop:
//   warp 0 lane 0   TMA producer: waits for a free stage, posts its byte
//                   count, loads the weight tile(s) and the activation rows;
//                   a task with a dependency loads its first weight tiles
//                   *before* it waits on the event, so the weight stream is
//                   already in flight when the dependency resolves;
//   warp 1 lane 0   MMA issuer: per task, waits for a free TMEM accumulator
//                   buffer, issues tcgen05.mma per full stage, frees each
//                   stage with tcgen05.commit, commits the accumulator;
//   warps 4..7      workers: the epilogue (tcgen05.ld from TMEM, stores,
//                   event releases) and every non-GEMM task; they sync among
//                   themselves with named barrier 1.
// Two TMEM accumulator buffers of 256 columns let the MMA of task i+1 run
// while the workers drain task i.
#pragma once

#include "et_device.cuh"

namespace et {

constexpr int kTaskRing = 4;      // dynamic-queue tasks handed from producer to consumers
constexpr int kWorkers = 128;     // warps 4..7
constexpr int kWorkerBar = 1;     // named barrier id of the worker group
constexpr int kAccBufCols = 256;  // TMEM columns per accumulator buffer

// One task as handed through the smem ring (dynamic schedules).
struct TaskMsg {
    int32_t type, a, b, c;  // type | (split << 8), then task-specific indices
    int32_t e, row0, rows, n;
};

// Per-CTA control block, after the stage ring and the SIMT scratch in smem.
struct Ctl {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t acc_full[2];
    uint64_t acc_empty[2];
    uint64_t tq_full[kTaskRing];
    uint64_t tq_empty[kTaskRing];
    uint64_t drain;
    TaskMsg tq[kTaskRing];
    uint32_t tmem_base;
    int32_t issued;    // stage fills posted by the producer (for the unwind)
    int32_t consumed;  // stage fills consumed by the MMA issuer
    int32_t flag;      // worker broadcast
    int32_t wflag[2];  // worker_wait decisions, double buffered
    int32_t scratch[16];
};

// Stage ring geometry: stage = [A0 16K][A1 16K][B nmax*128].
struct Stages {
    uint8_t* base;
    int n;
    int bytes;
    int b_off;
};

struct GemmTask {
    const CUtensorMap* a0;  // weight map, box 64 x 128
    const CUtensorMap* a1;  // second weight map (gate/up) or nullptr
    const CUtensorMap* b;   // activation map, box 64 x 16
    int a_row;              // first weight row
    int b_row;              // first activation row
    int kb0, nkb;           // k-blocks [kb0, kb0 + nkb), 64 elements each
    int n;                  // UMMA N: multiple of 16
    int kpack;              // k-blocks per stage when a1 == nullptr (1 or 2)
    const int* dep;         // wait *dep >= dep_target before activation loads
    int dep_target;
    int dep_where;
};

__device__ __forceinline__ int kpack_of(const GemmTask& t) { return t.a1 ? 1 : t.kpack; }

// ------------------------------------------------------------------ producer

// Issues every load of one GEMM task.  `it` counts stage fills over the
// whole launch (stage = it % n, phase = (it / n) & 1).  With a dependency,
// the weight tiles of the first min(units, stages) fills are posted first,
// then the event is awaited, then their activation rows follow.
__device__ __forceinline__ void load_acts(const GemmTask& t, const Stages& s, Ctl* ctl, uint32_t f,
                                          int u, uint64_t pol_b) {
    const int kp = kpack_of(t);
    const int st = static_cast<int>(f % s.n);
    const int nk = min(kp, t.nkb - u * kp);
    const uint32_t bbytes = static_cast<uint32_t>(t.n) * 128u;
    uint8_t* bb = s.base + st * s.bytes + s.b_off;
    for (int j = 0; j < nk; ++j)
        for (int i = 0; i < t.n / kBBoxRows; ++i)
            tma_load_2d(bb + j * bbytes + i * (kBBoxRows * 128), t.b, &ctl->full[st],
                        (t.kb0 + u * kp + j) * kBlockK, t.b_row + i * kBBoxRows, pol_b);
}

__device__ __forceinline__ bool post_weights(const GemmTask& t, const Stages& s, Ctl* ctl,
                                             uint32_t f, int u, const WaitCtx& wc,
                                             uint64_t pol_w) {
    const int kp = kpack_of(t);
    const int st = static_cast<int>(f % s.n);
    if (!mbar_wait(wc, &ctl->empty[st], ((f / s.n) & 1u) ^ 1u, kWhereEmpty)) return false;
    const int nk = min(kp, t.nkb - u * kp);
    const uint32_t bytes = (t.a1 ? 2u : static_cast<uint32_t>(nk)) * kABytes +
                           static_cast<uint32_t>(nk) * static_cast<uint32_t>(t.n) * 128u;
    mbar_arrive_expect_tx(&ctl->full[st], bytes);
    uint8_t* sb = s.base + st * s.bytes;
    const int kb = t.kb0 + u * kp;
    if (t.a1) {
        tma_load_2d(sb, t.a0, &ctl->full[st], kb * kBlockK, t.a_row, pol_w);
        tma_load_2d(sb + kABytes, t.a1, &ctl->full[st], kb * kBlockK, t.a_row, pol_w);
    } else {
        for (int j = 0; j < nk; ++j)
            tma_load_2d(sb + j * kABytes, t.a0, &ctl->full[st], (kb + j) * kBlockK, t.a_row, pol_w);
    }
    return true;
}

__device__ __forceinline__ bool produce_task(const GemmTask& t, const Stages& s, Ctl* ctl,
                                             uint32_t& it, const WaitCtx& wc, uint64_t pol_w,
                                             uint64_t pol_b) {
    const int units = ceil_div(t.nkb, kpack_of(t));
    const int pre = t.dep ? min(units, s.n) : 0;
    bool ok = true;
    int posted = 0;
    for (int u = 0; u < pre && ok; ++u) {  // weights first, ahead of the dependency
        ok = post_weights(t, s, ctl, it + u, u, wc, pol_w);
        if (ok) posted = u + 1;
    }
    if (ok && t.dep) {
        ok = ev_wait_geq(wc, t.dep, t.dep_target, t.dep_where);
        if (ok) {
            fence_proxy_async_global();  // rows written by other CTAs' generic stores
            for (int u = 0; u < pre; ++u) load_acts(t, s, ctl, it + u, u, pol_b);
        }
    }
    for (int u = pre; u < units && ok; ++u) {
        ok = post_weights(t, s, ctl, it + u, u, wc, pol_w);
        if (ok) {
            posted = u + 1;
            load_acts(t, s, ctl, it + u, u, pol_b);
        }
    }
    it += posted;
    ctl->issued = static_cast<int32_t>(it);
    return ok;
}

// ------------------------------------------------------------------ MMA issuer

// `it` counts consumed stage fills; `g` counts GEMM tasks (accumulator
// buffer = g % nbuf).  u_off is the column offset of the second accumulator.
__device__ __forceinline__ bool mma_task(const GemmTask& t, const Stages& s, Ctl* ctl, uint32_t& it,
                                         uint32_t& g, int nbuf, uint32_t u_off, uint32_t tmem,
                                         const WaitCtx& wc) {
    const uint32_t buf = g % nbuf, use = g / nbuf;
    if (!mbar_wait(wc, &ctl->acc_empty[buf], (use & 1u) ^ 1u, kWhereAcc)) return false;
    tc_fence_after();
    const int kp = kpack_of(t);
    const int units = ceil_div(t.nkb, kp);
    const uint32_t idesc = idesc_bf16_m128(t.n);
    const uint32_t bbytes = static_cast<uint32_t>(t.n) * 128u;
    const uint32_t acc0 = tmem + buf * kAccBufCols;
    const uint32_t acc1 = acc0 + u_off;
    for (int u = 0; u < units; ++u) {
        const int st = static_cast<int>(it % s.n);
        if (!mbar_wait(wc, &ctl->full[st], (it / s.n) & 1u, kWhereFull)) return false;
        it += 1;
        ctl->consumed = static_cast<int32_t>(it);
        tc_fence_after();
        const uint32_t sb = smem_u32(s.base + st * s.bytes);
        const int nk = min(kp, t.nkb - u * kp);
        for (int j = 0; j < nk; ++j) {
            const uint32_t a_s = sb + (t.a1 ? 0u : static_cast<uint32_t>(j) * kABytes);
            const uint32_t b_s = sb + s.b_off + static_cast<uint32_t>(j) * bbytes;
#pragma unroll
            for (int kk = 0; kk < kBlockK / 16; ++kk) {
                const uint32_t accumulate = (u > 0 || j > 0 || kk > 0) ? 1u : 0u;
                const uint64_t bd = sdesc_sw128(b_s + kk * 32);
                tc_mma_bf16(acc0, sdesc_sw128(a_s + kk * 32), bd, idesc, accumulate);
                if (t.a1)
                    tc_mma_bf16(acc1, sdesc_sw128(sb + kABytes + kk * 32), bd, idesc, accumulate);
            }
        }
        tc_commit(&ctl->empty[st]);
    }
    tc_commit(&ctl->acc_full[buf]);
    g += 1;
    return true;
}

// ------------------------------------------------------------------ workers

__device__ __forceinline__ void worker_sync() { named_bar_sync(kWorkerBar, kWorkers); }

// A bounded mbarrier wait taken by the whole worker group: one worker thread
// waits, the decision is broadcast, so all four worker warps always take the
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

// Wait for the accumulator of the workers' next GEMM task; returns its TMEM
// base (lane 0, first column of the buffer) through `acc`.
__device__ __forceinline__ bool epi_acquire(Ctl* ctl, uint32_t g, int nbuf, uint32_t tmem,
                                            const WaitCtx& wc, uint32_t& acc, uint32_t& seq) {
    const uint32_t buf = g % nbuf, use = g / nbuf;
    if (!worker_wait(ctl, &ctl->acc_full[buf], use & 1u, wc, kWhereAcc, seq)) return false;
    tc_fence_after();
    acc = tmem + buf * kAccBufCols;
    return true;
}

// The worker warp is done reading the accumulator buffer of task g.
__device__ __forceinline__ void epi_release(Ctl* ctl, uint32_t g, int nbuf) {
    tc_fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&ctl->acc_empty[g % nbuf]);
}

// ------------------------------------------------------------------ set-up / unwind

// Dynamic smem layout: [align 1024][stages x stage_bytes][scratch][Ctl].
__host__ __device__ constexpr int smem_bytes_for(int stages, int nmax, int scratch) {
    return 1024 + stages * stage_bytes(nmax) + scratch + static_cast<int>(sizeof(Ctl));
}

__device__ __forceinline__ Ctl* cta_setup(uint8_t* smem_raw, int stages, int nmax, int scratch,
                                          Stages& s, uint8_t** scratch_out) {
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    s.base = base;
    s.n = stages;
    s.bytes = stage_bytes(nmax);
    s.b_off = 2 * kABytes;
    *scratch_out = base + stages * s.bytes;
    Ctl* ctl = reinterpret_cast<Ctl*>(base + stages * s.bytes + scratch);
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kMaxStages; ++i) {
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
        ctl->issued = 0;
        ctl->consumed = 0;
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
__device__ __forceinline__ void cta_teardown(Ctl* ctl, const Stages& s, bool aborted_run) {
    __syncthreads();
    if (aborted_run && threadIdx.x == 32) {
        const uint64_t budget = 2000000ull;  // 2 ms per wait
        for (uint32_t c = static_cast<uint32_t>(ctl->consumed);
             c < static_cast<uint32_t>(ctl->issued); ++c)
            mbar_drain(&ctl->full[c % s.n], (c / s.n) & 1u, budget);
        tc_commit(&ctl->drain);
        mbar_drain(&ctl->drain, 0, budget);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if ((threadIdx.x >> 5) == 1) tmem_dealloc(ctl->tmem_base, kTmemCols);
}

// Stages that fit next to `scratch` bytes of SIMT scratch.
__host__ __device__ constexpr int stages_for(int nmax, int scratch) {
    return (kSmemLimit - 1024 - scratch - static_cast<int>(sizeof(Ctl))) / stage_bytes(nmax) >
                   kMaxStages
               ? kMaxStages
               : (kSmemLimit - 1024 - scratch - static_cast<int>(sizeof(Ctl))) / stage_bytes(nmax);
}

}  // namespace et
