// et_gemm.cuh -- one tiled GEMM task inside a persistent CTA:
//   D[128 weight rows, n token rows] = sum_k W[a_row.., k] * Act[b_row.., k]
// with the weight tile on the UMMA M side ("swap-AB": decode-sized token
// counts sit on N, which may be as small as 16).
//
// Roles (warp specialised inside one task; the whole CTA meets at the end):
//   warp 0 lane 0  TMA producer: waits for a free stage, posts the byte count,
//                  loads the weight tile(s) and the activation rows;
//   warp 1 lane 0  MMA issuer: waits for a full stage, issues tcgen05.mma into
//                  TMEM, commits the stage back to the producer;
//   warps 4..7     epilogue: wait for the accumulator, tcgen05.ld, then the
//                  task's own store / event logic.
// A task with a dependency (an event counter that another task releases)
// loads its first weight tiles *before* it waits, so the weight stream is
// already in flight when the dependency resolves.
#pragma once

#include "et_device.cuh"

namespace et {

// Per-CTA control block, placed after the stage ring in dynamic smem.
struct Ctl {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t acc_full;
    uint64_t drain;
    uint32_t tmem_base;
    int32_t fail;          // a wait of this CTA failed during the current task
    int32_t issued_total;  // producer's running stage-fill count
    int32_t flag;          // scratch broadcast
    int4 task;             // current task
    int32_t scratch[64];   // small broadcast values of SIMT tasks
};

// Stage ring geometry.
struct Ring {
    uint8_t* base;
    int stages;
    int stage_bytes;
    int b_off;  // byte offset of the activation region inside a stage
};

// Per-role running pipeline state (kept in registers of the role's thread).
struct Pipe {
    uint32_t cursor = 0;      // stage fills issued (producer) / consumed (MMA)
    uint32_t phase_bits = 0;  // per-stage phase parity
    uint32_t acc_phase = 0;   // epilogue: parity of acc_full
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

__device__ __forceinline__ int units_of(const GemmTask& t) {
    const int kp = t.a1 ? 1 : t.kpack;
    return ceil_div(t.nkb, kp);
}

// ------------------------------------------------------------------ producer

static __device__ __noinline__ bool gemm_producer(const GemmTask& t, const Ring& r, Ctl* ctl, Pipe& pp,
                                           const WaitCtx& wc, uint64_t pol_w, uint64_t pol_b) {
    const int kp = t.a1 ? 1 : t.kpack;
    const int units = ceil_div(t.nkb, kp);
    const uint32_t bbytes = static_cast<uint32_t>(t.n) * 128u;
    const int pre = t.dep ? min(units, r.stages) : 0;
    bool ok = true;
    int issued = 0;

    auto stage_of = [&](int u) { return static_cast<int>((pp.cursor + u) % r.stages); };
    // wait for a free stage, post its byte count, load the weight tile(s)
    auto post_weights = [&](int u) -> bool {
        const int st = stage_of(u);
        if (!mbar_wait(wc, &ctl->empty[st], ((pp.phase_bits >> st) & 1u) ^ 1u, kWhereEmpty))
            return false;
        pp.phase_bits ^= 1u << st;
        const int nk = min(kp, t.nkb - u * kp);
        const uint32_t bytes =
            (t.a1 ? 2u : static_cast<uint32_t>(nk)) * kABytes + static_cast<uint32_t>(nk) * bbytes;
        mbar_arrive_expect_tx(&ctl->full[st], bytes);
        uint8_t* sb = r.base + st * r.stage_bytes;
        const int kb = t.kb0 + u * kp;
        if (t.a1) {
            tma_load_2d(sb, t.a0, &ctl->full[st], kb * kBlockK, t.a_row, pol_w);
            tma_load_2d(sb + kABytes, t.a1, &ctl->full[st], kb * kBlockK, t.a_row, pol_w);
        } else {
            for (int j = 0; j < nk; ++j)
                tma_load_2d(sb + j * kABytes, t.a0, &ctl->full[st], (kb + j) * kBlockK, t.a_row,
                            pol_w);
        }
        return true;
    };
    auto load_acts = [&](int u) {
        const int st = stage_of(u);
        const int nk = min(kp, t.nkb - u * kp);
        uint8_t* sb = r.base + st * r.stage_bytes + r.b_off;
        const int kb = t.kb0 + u * kp;
        for (int j = 0; j < nk; ++j)
            for (int i = 0; i < t.n / kBBoxRows; ++i)
                tma_load_2d(sb + j * bbytes + i * (kBBoxRows * 128), t.b, &ctl->full[st],
                            (kb + j) * kBlockK, t.b_row + i * kBBoxRows, pol_b);
    };

    for (int u = 0; u < pre; ++u) {
        if (!post_weights(u)) { ok = false; break; }
        ++issued;
    }
    if (ok && t.dep) {
        ok = ev_wait_geq(wc, t.dep, t.dep_target, t.dep_where);
        if (ok) fence_proxy_async_global();
    }
    if (ok)
        for (int u = 0; u < pre; ++u) load_acts(u);
    for (int u = pre; ok && u < units; ++u) {
        if (!post_weights(u)) { ok = false; break; }
        ++issued;
        load_acts(u);
    }
    pp.cursor += issued;
    ctl->issued_total = static_cast<int32_t>(pp.cursor);
    return ok;
}

// ------------------------------------------------------------------ MMA issuer

static __device__ __noinline__ bool gemm_mma(const GemmTask& t, const Ring& r, Ctl* ctl, Pipe& pm,
                                      uint32_t tmem_base, const WaitCtx& wc) {
    tc_fence_after();
    const int kp = t.a1 ? 1 : t.kpack;
    const int units = ceil_div(t.nkb, kp);
    const uint32_t idesc = idesc_bf16_m128(t.n);
    const uint32_t bbytes = static_cast<uint32_t>(t.n) * 128u;
    const uint32_t acc0 = tmem_base;
    const uint32_t acc1 = tmem_base + kAcc1Col;
    for (int u = 0; u < units; ++u) {
        const int st = static_cast<int>(pm.cursor % r.stages);
        if (!mbar_wait(wc, &ctl->full[st], (pm.phase_bits >> st) & 1u, kWhereFull)) return false;
        pm.phase_bits ^= 1u << st;
        pm.cursor += 1;
        tc_fence_after();
        const uint32_t sb = smem_u32(r.base + st * r.stage_bytes);
        const int nk = min(kp, t.nkb - u * kp);
        for (int j = 0; j < nk; ++j) {
            const uint32_t a_s = sb + (t.a1 ? 0u : static_cast<uint32_t>(j) * kABytes);
            const uint32_t b_s = sb + r.b_off + static_cast<uint32_t>(j) * bbytes;
#pragma unroll
            for (int kk = 0; kk < kBlockK / 16; ++kk) {
                const uint32_t accumulate = (u > 0 || j > 0 || kk > 0) ? 1u : 0u;
                const uint64_t bd = sdesc_sw128(b_s + kk * 32);
                tc_mma_bf16(acc0, sdesc_sw128(a_s + kk * 32), bd, idesc, accumulate);
                if (t.a1) tc_mma_bf16(acc1, sdesc_sw128(sb + kABytes + kk * 32), bd, idesc, accumulate);
            }
        }
        tc_commit(&ctl->empty[st]);  // stage is free once these MMAs finish
    }
    tc_commit(&ctl->acc_full);
    return true;
}

// ------------------------------------------------------------------ one task, whole CTA

// Runs the roles of one GEMM task; `epi(q, lane)` is executed by the 4
// epilogue warps (q = 0..3 is the TMEM lane quarter) once the accumulator is
// complete.  Returns false (on every thread) if any wait of this CTA failed.
template <class Epi>
__device__ __forceinline__ bool run_gemm_task(const GemmTask& t, Ctl* ctl, const Ring& r,
                                              Pipe& pipe, uint32_t tmem_base, const WaitCtx& wc,
                                              uint64_t pol_w, uint64_t pol_b, Epi&& epi) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 0) {
        if (lane == 0 && !gemm_producer(t, r, ctl, pipe, wc, pol_w, pol_b)) ctl->fail = 1;
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0 && !gemm_mma(t, r, ctl, pipe, tmem_base, wc)) ctl->fail = 1;
        __syncwarp();
    } else if (warp >= kEpiWarp0) {
        const bool ok = mbar_wait(wc, &ctl->acc_full, pipe.acc_phase, kWhereAcc);
        pipe.acc_phase ^= 1u;
        if (ok) {
            tc_fence_after();
            epi(warp - kEpiWarp0, lane);
        } else {
            ctl->fail = 1;
        }
        tc_fence_before();
    }
    __syncthreads();
    return ctl->fail == 0;
}

// After a failed task: let this CTA's own TMA copies and MMAs land (bounded,
// without raising) so that the CTA can release TMEM and exit cleanly.
// Called by every thread; the MMA thread does the waiting.
__device__ __forceinline__ void drain_after_failure(Ctl* ctl, const Ring& r, Pipe& pipe) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == 1 && lane == 0) {
        const uint64_t budget = 2000000ull;  // 2 ms per wait
        const uint32_t issued = static_cast<uint32_t>(ctl->issued_total);
        while (pipe.cursor < issued) {
            const int st = static_cast<int>(pipe.cursor % r.stages);
            mbar_drain(&ctl->full[st], (pipe.phase_bits >> st) & 1u, budget);
            pipe.phase_bits ^= 1u << st;
            pipe.cursor += 1;
        }
        tc_commit(&ctl->drain);
        mbar_drain(&ctl->drain, 0, budget);
    }
    __syncwarp();
    __syncthreads();
}

// Shared-memory set-up common to all kernels: ring, control block, barriers,
// TMEM.  Returns the control block; `ring` is filled in.
__device__ __forceinline__ Ctl* cta_setup(uint8_t* smem_raw, int stages, int nmax, Ring& ring) {
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    ring.base = base;
    ring.stages = stages;
    ring.stage_bytes = stage_bytes(nmax);
    ring.b_off = 2 * kABytes;
    Ctl* ctl = reinterpret_cast<Ctl*>(base + stages * ring.stage_bytes);
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kMaxStages; ++i) {
            mbar_init(&ctl->full[i], 1);
            mbar_init(&ctl->empty[i], 1);
        }
        mbar_init(&ctl->acc_full, 1);
        mbar_init(&ctl->drain, 1);
        ctl->fail = 0;
        ctl->issued_total = 0;
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

__device__ __forceinline__ void cta_teardown(Ctl* ctl) {
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if ((threadIdx.x >> 5) == 1) tmem_dealloc(ctl->tmem_base, kTmemCols);
}

// Dynamic shared memory a kernel needs for `stages` stages of width nmax.
__host__ __device__ constexpr int smem_bytes_for(int stages, int nmax) {
    return 1024 /*alignment slack*/ + stages * stage_bytes(nmax) + static_cast<int>(sizeof(Ctl));
}

}  // namespace et
