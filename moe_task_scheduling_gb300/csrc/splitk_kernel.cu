// splitk_kernel.cu -- split-K GEMM whose partial sums meet through event
// counters instead of a second kernel:
//   Y[M,N] = bf16( sum_{s < split} X[:, K_s] Wt[:, K_s]^T )
// Static schedule (task t runs on CTA t mod grid; every role walks the same
// task list):
//   [0, G)        TILE (mt, nt, s): fp32 partial of a 256 x 128 output tile over
//                 K chunk s (bf16 Y directly when split == 1); releases
//                 ev[mt][nt]
//   [G, G + R)    REDUCE (q, nt), split > 1 and M > 32 only: waits ev[tile] >=
//                 split, then sums rows [32q, 32q + 32) of the tile's partials
//                 in chunk order and stores bf16 Y.  With M <= 32 the TILE
//                 task that completes ev[tile] sums it instead (same order),
//                 so no task polls for it.
// Every wait is on a lower task index, and the launch is cooperative (every
// CTA resident), so the schedule cannot deadlock; the reduction of one tile is
// spread over many CTAs instead of falling on the last arriver.  The last CTA
// out returns the tile counters to zero.  M stays symbolic: it may be read
// from device memory, and the same compiled kernel serves every M up to M_max.
//
// Source: "Prompt Boundary-Aware Scheduling with Event Tensors for Dynamic
// Kernels" -- the split-K summation example, where the reduction is gated by
// an event over the producing tiles rather than by a kernel boundary.
#include "et_gemm.cuh"

namespace et {

struct SplitKTile {
    int s, nt, mt, rows, n;
};

__device__ __forceinline__ SplitKTile splitk_tile(int task, int split, int NT, int M) {
    SplitKTile t;
    t.s = task % split;
    const int rest = task / split;
    t.nt = rest % NT;
    t.mt = rest / NT;
    t.rows = min(kWideNMax, M - t.mt * kWideNMax);
    t.n = (t.rows + 15) / 16 * 16;
    return t;
}

__global__ void __launch_bounds__(kThreads, 1)
splitk_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
              const __grid_constant__ CUtensorMap tm_x64, const __grid_constant__ SplitKArgs p) {
    extern __shared__ uint8_t smem_raw[];
    const uint64_t t_start = globaltimer_ns();
    Ring ring;
    uint8_t* scratch;
    Ctl* ctl = cta_setup(smem_raw, 0, ring, &scratch);
    if (threadIdx.x == 0) trace_put(p.trace, p.trace_cap, 0, 2, 0, 0, t_start, globaltimer_ns());
    const WaitCtx wc{p.hdr, p.timeout_ns};
    const uint32_t tmem = ctl->tmem_base;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    int M = p.M_host;
    if (p.d_M) M = *reinterpret_cast<const volatile int32_t*>(p.d_M);
    if (M < 0 || M > p.M_max) {
        if (blockIdx.x == 0 && threadIdx.x == 0) raise_error(wc, ET_ERR_BOUNDS, kWhereBoundsT);
        M = 0;
    }
    const int N = p.N, split = p.split;
    const int MT = ceil_div(M, kWideNMax), NT = N / kTileM;
    const int kbs = p.K / kBlockK / split;
    const int total = MT * NT * split;
    constexpr int kRedRows = 32;  // rows per reduce task
    // a tile of at most 32 rows is summed by the split that completes its
    // counter (no reduce task polls for it); taller tiles spread their rows
    // over reduce tasks
    const bool last_arriver = split > 1 && M <= kRedRows;
    const int n_red = (split > 1 && !last_arriver) ? ceil_div(M, kRedRows) * NT : 0;

    auto gemm_of = [&](const SplitKTile& t) {
        return GemmTask{&tm_w, nullptr, &tm_x, p.b_wide ? &tm_x64 : nullptr, t.nt * kTileM,
                        t.mt * kWideNMax, t.s * kbs, kbs, t.n, nullptr, 0, 0};
    };

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first(), pol_b = policy_evict_last();
            int task = blockIdx.x;
            auto next = [&](GemmTask& g) {  // this CTA's next tile task
                if (task >= total) return false;
                g = gemm_of(splitk_tile(task, split, NT, M));
                task += gridDim.x;
                return true;
            };
            produce_static(next, ring, ctl, wc, pol_w, pol_b);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            MmaState ms;
            for (int task = blockIdx.x; task < total; task += gridDim.x) {
                auto ftr = [&](int u, uint64_t tp, uint64_t tl) {
                    trace_put(p.trace, p.trace_cap, kTaskSplitK, 5, task, u, tp, tl);
                };
                if (!mma_task(gemm_of(splitk_tile(task, split, NT, M)), ring, ctl, ms, tmem, wc, ftr))
                    break;
            }
        }
        __syncwarp();
    } else if (warp >= kEpiWarp0) {
        const int q = warp & 3, half = (warp - kEpiWarp0) >> 2;  // TMEM lane quadrant, column half
        const int wtid = threadIdx.x - kEpiWarp0 * 32;
        EpiState es;
        for (int task = blockIdx.x; task < total + n_red; task += gridDim.x) {
            const uint64_t tw = p.trace ? globaltimer_ns() : 0;
            if (task >= total) {  // REDUCE: row slice qs of tile column nt
                const int r = task - total, nt = r % NT, qs = r / NT;
                const int r0 = qs * kRedRows, r1 = min(M, r0 + kRedRows), mt = r0 / kWideNMax;
                if (wtid == 0)
                    ctl->flag = ev_wait_geq(wc, p.ev + mt * NT + nt, split, kWhereY) ? 1 : 0;
                worker_sync();
                if (!ctl->flag) break;
                reduce_slice(p.partial, static_cast<size_t>(p.M_max) * N, N, split, r0, r1,
                             nt * kTileM, p.Y, N);
                if (wtid == 0) trace_put(p.trace, p.trace_cap, kTaskReduce, 1, task, 0, tw, globaltimer_ns());
                continue;
            }
            const SplitKTile t = splitk_tile(task, split, NT, M);
            uint32_t acc, acc1;
            if (!epi_acquire(ctl, es, false, t.n, tmem, wc, acc, acc1)) break;
            if (wtid == 0) trace_put(p.trace, p.trace_cap, kTaskSplitK, 6, task, 0, tw, globaltimer_ns());
            const int col = t.nt * kTileM + q * 32 + lane;
            const uint32_t lane_base = acc + (static_cast<uint32_t>(q * 32) << 16);
            const size_t m0 = static_cast<size_t>(t.mt) * kWideNMax;
            for (int c0 = half * 16; c0 < t.n; c0 += 32) {
                float v[16];
                tmem_ld16(lane_base + c0, v);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    if (c0 + c >= t.rows) continue;
                    const size_t m = m0 + c0 + c;
                    if (split == 1)
                        p.Y[m * N + col] = __float2bfloat16_rn(v[c]);
                    else
                        p.partial[(static_cast<size_t>(t.s) * p.M_max + m) * N + col] = v[c];
                }
            }
            epi_release(ctl, es, false, t.n);
            if (last_arriver) {  // the split that completes the tile sums its partials
                int* ev = p.ev + t.mt * NT + t.nt;
                worker_sync();
                if (wtid == 0) {
                    __threadfence();
                    ctl->flag = (atom_acq_rel_add(ev, 1) == split - 1) ? 1 : 0;
                }
                worker_sync();
                const bool last = ctl->flag != 0;
                worker_sync();  // the flag is read before any later task writes it
                if (last) {
                    if (wtid == 0) *ev = 0;  // every split arrived: reset for the next call
                    reduce_slice4(p.partial, static_cast<size_t>(p.M_max) * N, N, split,
                                  static_cast<int>(m0), static_cast<int>(m0) + t.rows,
                                  t.nt * kTileM, p.Y, N);
                }
            } else if (split > 1) {  // the partial is stored: count it on the tile's event
                worker_sync();
                if (wtid == 0) {
                    __threadfence();
                    red_release_add(p.ev + t.mt * NT + t.nt, 1);
                }
            }
            if (wtid == 0) trace_put(p.trace, p.trace_cap, kTaskSplitK, 1, task, 0, tw, globaltimer_ns());
        }
    }

    const uint64_t t_exit = globaltimer_ns();
    const bool aborted_run = ld_relaxed(&p.hdr->abort) != 0;
    cta_teardown(ctl, aborted_run);
    __syncthreads();
    if (threadIdx.x == 0) {
        trace_put(p.trace, p.trace_cap, 0, 3, 0, 0, t_exit, globaltimer_ns());
        __threadfence();
        if (atomicAdd(&p.hdr->exit_count, 1) == static_cast<int>(gridDim.x) - 1) {
            // the tile counters go back to zero (all of them after an abort)
            const int n_ev = ld_relaxed(&p.hdr->abort) != 0 ? ceil_div(p.M_max, kWideNMax) * NT
                                                           : (split > 1 ? MT * NT : 0);
            for (int i = 0; i < n_ev; ++i) p.ev[i] = 0;
            p.hdr->abort = 0;
            __threadfence();
            p.hdr->exit_count = 0;
        }
    }
}

// ------------------------------------------------------------------ Cluster Launch Control

// The same GEMM with the hardware as the work queue ("Megakernels ch. 5 -
// Event Tensor et le dynamisme", section 5.5: Blackwell's Cluster Launch
// Control lets a running CTA take over the work of a CTA that has not started).
// The grid has one CTA per TILE task (all M tiles up to M_max); a running CTA
// asks the hardware to cancel a CTA that has not launched yet and runs that
// CTA's task itself, so one CTA's set-up (TMEM, barriers, tensor maps) serves
// several tasks while the launch hardware does the balancing, and other work
// on the GPU can interleave (no cooperative launch).  No task waits on
// another: the task that completes a tile's counter sums the tile's partials
// in split order (the last arriver) and returns the counter to zero.

constexpr int kClcScratch = 64;  // smem: the 16-byte cancel response, its mbarrier

// reduce_slice for one whole tile on one CTA: two float4 columns per thread at
// a time, every split's loads in flight (split <= 8), the same sum order.
static __device__ __noinline__ void reduce_tile2(const float* part, size_t sstride, int ld, int split,
                                             int r0, int r1, int col0, bf16* Y, int ldy) {
    constexpr int kMax = 8, kV = kTileM / 4;  // float4 columns a row
    const int nv = (r1 - r0) * kV, wt = static_cast<int>(threadIdx.x) - kEpiWarp0 * 32;
    for (int v0 = wt; v0 < nv; v0 += 2 * kWorkers) {
        float4 q[2][kMax];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int v = v0 + u * kWorkers;
            if (v >= nv) continue;
            const float* src = part + static_cast<size_t>(r0 + v / kV) * ld + col0 + (v % kV) * 4;
#pragma unroll
            for (int s = 0; s < kMax; ++s)
                if (s < split) q[u][s] = __ldcg(reinterpret_cast<const float4*>(src + s * sstride));
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int v = v0 + u * kWorkers;
            if (v >= nv) continue;
            float4 acc = q[u][0];
#pragma unroll
            for (int s = 1; s < kMax; ++s)
                if (s < split) {
                    acc.x = acc.x + q[u][s].x;
                    acc.y = acc.y + q[u][s].y;
                    acc.z = acc.z + q[u][s].z;
                    acc.w = acc.w + q[u][s].w;
                }
            __nv_bfloat162 o[2] = {__floats2bfloat162_rn(acc.x, acc.y),
                                   __floats2bfloat162_rn(acc.z, acc.w)};
            *reinterpret_cast<uint2*>(Y + static_cast<size_t>(r0 + v / kV) * ldy + col0 +
                                      (v % kV) * 4) = *reinterpret_cast<const uint2*>(o);
        }
    }
}

__device__ __forceinline__ void clc_try_cancel(void* response, uint64_t* bar) {
    asm volatile(
        "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 "
        "[%0], [%1];" ::"r"(smem_u32(response)),
        "r"(smem_u32(bar))
        : "memory");
}

// The cancelled CTA's x index, or -1 when the request cancelled nothing (no
// CTA left to launch).
__device__ __forceinline__ int clc_result(const void* response) {
    uint32_t ok, x = 0;
    asm volatile(
        "{\n\t.reg .b128 r;\n\t.reg .pred p;\n\t"
        "ld.shared.b128 r, [%2];\n\t"
        "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t"
        "@p clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, r;\n\t}"
        : "=r"(ok), "+r"(x)
        : "r"(smem_u32(response))
        : "memory");
    return ok ? static_cast<int>(x) : -1;
}

__global__ void __launch_bounds__(kThreads, 1)
splitk_clc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                  const __grid_constant__ CUtensorMap tm_x64, const __grid_constant__ SplitKArgs p) {
    extern __shared__ uint8_t smem_raw[];
    Ring ring;
    uint8_t* scratch;
    Ctl* ctl = cta_setup(smem_raw, kClcScratch, ring, &scratch);
    uint64_t* clc_bar = reinterpret_cast<uint64_t*>(scratch + 16);
    if (threadIdx.x == 0) {
        mbar_init(clc_bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    const WaitCtx wc{p.hdr, p.timeout_ns};
    const uint32_t tmem = ctl->tmem_base;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    int M = p.M_host;
    if (p.d_M) M = *reinterpret_cast<const volatile int32_t*>(p.d_M);
    if (M < 0 || M > p.M_max) {
        if (blockIdx.x == 0 && threadIdx.x == 0) raise_error(wc, ET_ERR_BOUNDS, kWhereBoundsT);
        M = 0;
    }
    const int N = p.N, split = p.split;
    const int MT = ceil_div(M, kWideNMax), NT = N / kTileM;
    const int kbs = p.K / kBlockK / split;

    auto gemm_of = [&](const SplitKTile& t) {
        return GemmTask{&tm_w, nullptr, &tm_x, p.b_wide ? &tm_x64 : nullptr, t.nt * kTileM,
                        t.mt * kWideNMax, t.s * kbs, kbs, t.n, nullptr, 0, 0};
    };

    if (warp == 0) {
        if (lane == 0) {  // producer: this CTA's task, then the tasks it cancels
            const uint64_t pol_w = policy_evict_first(), pol_b = policy_evict_last();
            ProdState ps;
            int task = static_cast<int>(blockIdx.x), owned = 0, sent = 0, asked = 0;
            for (;;) {
                if (task >= 0) {
                    ++owned;  // counted whether it runs or is skipped
                    const SplitKTile t = splitk_tile(task, split, NT, M);
                    if (t.mt >= MT || aborted(wc)) task = -1;  // nothing to compute
                }
                // hand the task (or the end, -1) to the MMA issuer and the workers
                const int slot = sent % kTaskRing;
                if (!mbar_wait(wc, &ctl->tq_empty[slot], ((sent / kTaskRing) & 1) ^ 1, kWhereQueue))
                    break;
                ctl->tq[slot].type = task;
                mbar_arrive(&ctl->tq_full[slot]);
                ++sent;
                if (task < 0) break;
                // ask for the next task now; the answer arrives while this one loads
                mbar_arrive_expect_tx(clc_bar, 16);
                clc_try_cancel(scratch, clc_bar);
                const bool ok = produce_task(gemm_of(splitk_tile(task, split, NT, M)), ring, ctl, ps,
                                             wc, pol_w, pol_b);
                // the response is written asynchronously: wait for it even after an abort
                // (bounded by the time limit only)
                const uint64_t t0 = globaltimer_ns();
                bool got = true;
                while (!mbar_try_wait(clc_bar, asked & 1))
                    if (globaltimer_ns() - t0 > p.timeout_ns) {
                        raise_error(wc, ET_ERR_TIMEOUT, kWhereQueue);
                        got = false;
                        break;
                    }
                ++asked;
                task = got ? clc_result(scratch) : -1;
                if (!ok && task >= 0) {  // cancelled, but this CTA stops: count it as skipped
                    ++owned;
                    task = -1;
                }
            }
            ctl->scratch[0] = owned;
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            MmaState ms;
            for (int i = 0;; ++i) {
                const int slot = i % kTaskRing;
                if (!mbar_wait(wc, &ctl->tq_full[slot], (i / kTaskRing) & 1, kWhereQueue)) break;
                const int task = ctl->tq[slot].type;
                mbar_arrive(&ctl->tq_empty[slot]);
                if (task < 0) break;
                if (!mma_task(gemm_of(splitk_tile(task, split, NT, M)), ring, ctl, ms, tmem, wc))
                    break;
            }
        }
        __syncwarp();
    } else if (warp >= kEpiWarp0) {
        const int q = warp & 3, half = (warp - kEpiWarp0) >> 2;  // TMEM lane quadrant, column half
        const int wtid = threadIdx.x - kEpiWarp0 * 32;
        EpiState es;
        for (int i = 0;; ++i) {
            const int slot = i % kTaskRing;
            if (!worker_wait(ctl, &ctl->tq_full[slot], (i / kTaskRing) & 1, wc, kWhereQueue, es.seq))
                break;
            const int task = ctl->tq[slot].type;
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->tq_empty[slot]);
            if (task < 0) break;
            const SplitKTile t = splitk_tile(task, split, NT, M);
            uint32_t acc, acc1;
            if (!epi_acquire(ctl, es, false, t.n, tmem, wc, acc, acc1)) break;
            const int col = t.nt * kTileM + q * 32 + lane;
            const uint32_t lane_base = acc + (static_cast<uint32_t>(q * 32) << 16);
            const size_t m0 = static_cast<size_t>(t.mt) * kWideNMax;
            for (int c0 = half * 16; c0 < t.n; c0 += 32) {
                float v[16];
                tmem_ld16(lane_base + c0, v);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    if (c0 + c >= t.rows) continue;
                    const size_t m = m0 + c0 + c;
                    if (split == 1)
                        p.Y[m * N + col] = __float2bfloat16_rn(v[c]);
                    else
                        p.partial[(static_cast<size_t>(t.s) * p.M_max + m) * N + col] = v[c];
                }
            }
            epi_release(ctl, es, false, t.n);
            if (split > 1) {  // the partial is stored: the last of the tile's splits sums them
                int* ev = p.ev + t.mt * NT + t.nt;
                worker_sync();
                if (wtid == 0) {
                    __threadfence();
                    ctl->flag = (atom_acq_rel_add(ev, 1) == split - 1) ? 1 : 0;
                }
                worker_sync();
                if (ctl->flag) {
                    if (wtid == 0) *ev = 0;  // every split arrived: reset for the next call
                    if (split <= 8)
                        reduce_tile2(p.partial, static_cast<size_t>(p.M_max) * N, N, split,
                                     static_cast<int>(m0), static_cast<int>(m0) + t.rows,
                                     t.nt * kTileM, p.Y, N);
                    else
                        reduce_slice4(p.partial, static_cast<size_t>(p.M_max) * N, N, split,
                                      static_cast<int>(m0), static_cast<int>(m0) + t.rows,
                                      t.nt * kTileM, p.Y, N);
                }
                worker_sync();
            }
        }
    }

    const bool aborted_run = ld_relaxed(&p.hdr->abort) != 0;
    cta_teardown(ctl, aborted_run);
    __syncthreads();
    if (threadIdx.x == 0) {
        // every task of the grid is counted once, by the CTA that ran or skipped it;
        // the count that reaches the grid size belongs to the last CTA out
        const int owned = ctl->scratch[0];
        __threadfence();
        if (atomicAdd(&p.hdr->exit_count, owned) + owned == static_cast<int>(gridDim.x)) {
            if (ld_relaxed(&p.hdr->abort) != 0) {  // counters an aborted launch may have left
                const int n_ev = ceil_div(p.M_max, kWideNMax) * NT;
                for (int i = 0; i < n_ev; ++i) p.ev[i] = 0;
            }
            p.hdr->abort = 0;
            __threadfence();
            p.hdr->exit_count = 0;
        }
    }
}

int splitk_smem_bytes() { return smem_bytes_for(0); }
int splitk_clc_smem_bytes() { return smem_bytes_for(kClcScratch); }

cudaError_t launch_splitk_clc(const SplitKArgs& a, const CUtensorMap* maps, int grid, int smem,
                              cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, splitk_clc_kernel, maps[0], maps[1], maps[2], a);
}

cudaError_t prepare_splitk_clc(int smem) {
    return cudaFuncSetAttribute(splitk_clc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem);
}

cudaError_t launch_splitk(const SplitKArgs& a, const CUtensorMap* maps, int grid, int smem,
                          cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, splitk_kernel, maps[0], maps[1], maps[2], a);
}

cudaError_t prepare_splitk(int smem) {
    return cudaFuncSetAttribute(splitk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

}  // namespace et
