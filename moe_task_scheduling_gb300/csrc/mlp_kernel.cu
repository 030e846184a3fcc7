// mlp_kernel.cu -- dense dependent MLP chain under a STATIC schedule:
//   xhat = bf16(x * rsqrt(mean(x^2) + eps) * gamma)
//   h    = bf16(silu(xhat Wg^T) * (xhat Wu^T))
//   out  = bf16(h Wd^T)
// Tasks are bound to CTAs by index (task i runs on CTA i mod grid, in index
// order) -- no queue, no atomics for distribution.  Index order is
//   [0, NR)                 NORM i      row i (the whole worker group); releases ev_norm
//   [NR, NR + MT*FT*KC)     GATEUP m,f,c waits ev_norm >= NR; with a K split (small
//                                       batches: K chunks c) stores fp32 partials, and
//                                       the chunk that completes ev_gu[m][f] sums them;
//                                       then releases ev_h[m][chunk(f)]
//   [.., + MT*S*HT)         DOWN m,s,n  waits ev_h[m][s] >= F-tiles per chunk;
//                                       with a split, stores an fp32 partial and
//                                       releases ev_y[m][n]
//   [.., + ceil(B/32)*HT)   REDUCE q,n  (split only) waits ev_y[m][n] >= S, sums
//                                       rows 32q .. of the partials in chunk order
// so every wait is on a lower index, which a resident CTA reaches first (the
// launch is cooperative: all CTAs are resident).  The targets (NR, F-tiles
// per chunk) are computed on the device from the batch size, which may itself
// be read from device memory.
//
// Source: "Prompt Boundary-Aware Scheduling with Event Tensors for Dynamic
// Kernels" -- static scheduling is the right choice for predictable dense
// work; events still replace kernel boundaries between dependent tiles.
#include "et_gemm.cuh"

namespace et {

constexpr int kNormRows = 1;  // rows per NORM task (the whole worker group takes a row)

constexpr int kRedRows = 32;  // rows per REDUCE task

struct MlpPlan {
    int B, NR, MT, FT, HT, S, KC, n_gu, n_dn, n_red, total;
};

struct MlpTile {
    int kind;  // 0 norm, 1 gate/up, 2 down, 3 reduce
    int i, mt, ft, kc, s, ht, rows, n;
};

// Task index -> task (see the order above).  The down tiles come after
// every gate/up tile: placed right behind their own chunk's gate/up tiles
// they were measured slower (88-90 -> 100-113 us at B = 1..8): a down tile
// that waits for its chunk stalls its CTA's in-order sequence, and with it
// gate/up tiles other chunks wait for.
__device__ __forceinline__ MlpTile mlp_tile(const MlpPlan& P, int task) {
    MlpTile t{};
    if (task < P.NR) {
        t.kind = 0;
        t.i = task;
        return t;
    }
    if (task >= P.NR + P.n_gu + P.n_dn) {
        t.kind = 3;
        t.i = task - P.NR - P.n_gu - P.n_dn;
        t.ht = t.i % P.HT;
        t.s = t.i / P.HT;  // row slice
        return t;
    }
    if (task < P.NR + P.n_gu) {
        t.kind = 1;
        t.i = task - P.NR;
        t.kc = t.i % P.KC;  // the K chunks of one tile run on neighbouring CTAs
        t.mt = (t.i / P.KC) / P.FT;
        t.ft = (t.i / P.KC) % P.FT;
    } else {
        t.kind = 2;
        t.i = task - P.NR - P.n_gu;
        t.mt = t.i / (P.S * P.HT);
        const int rem = t.i % (P.S * P.HT);
        t.s = rem / P.HT;
        t.ht = rem % P.HT;
    }
    t.rows = min(kWideNMax, P.B - t.mt * kWideNMax);
    t.n = (t.rows + 15) / 16 * 16;
    return t;
}

// RMSNorm of row i by the whole worker group: each thread takes every 256th
// 16-byte vector of the row (up to four loads in flight), so a cold row costs
// about one memory round trip (one warp walking a 4096-wide row load after
// load took 9-13 us, and every gate/up tile waits for the norm).  The sum of
// squares meets through shared memory (warp partials added in warp order).
__device__ __forceinline__ void norm_row(const MlpArgs& p, int row, Ctl* ctl) {
    const int wt = static_cast<int>(threadIdx.x) - kEpiWarp0 * 32, lane = wt & 31;
    const int H = p.H, nv = H / 8;  // 16-byte vectors a row
    const uint4* xr = reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(row) * H);
    const uint4* gr = reinterpret_cast<const uint4*>(p.gamma);
    for (int c = wt * 8; c < nv; c += kWorkers * 8)  // gamma, one 128-byte line a prefetch
        asm volatile("prefetch.global.L2 [%0];" ::"l"(gr + c) : "memory");
    float ss = 0.0f;
    for (int c0 = wt; c0 < nv; c0 += kWorkers * 4) {
        uint4 raw[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (c0 + u * kWorkers < nv) raw[u] = __ldg(xr + c0 + u * kWorkers);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (c0 + u * kWorkers >= nv) continue;
            const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&raw[u]);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 f = __bfloat1622float2(b2[q]);
                ss = fmaf(f.x, f.x, ss);
                ss = fmaf(f.y, f.y, ss);
            }
        }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    float* part = reinterpret_cast<float*>(ctl->scratch);  // [8] warp partials
    if (lane == 0) part[wt >> 5] = ss;
    worker_sync();
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < kWorkers / 32; ++w) tot += part[w];
    const float rs = rsqrtf(tot / static_cast<float>(H) + p.eps);
    uint4* outr = reinterpret_cast<uint4*>(p.xhat + static_cast<size_t>(row) * H);
    for (int c0 = wt; c0 < nv; c0 += kWorkers * 4) {
        uint4 raw[4], graw[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (c0 + u * kWorkers < nv) {
                raw[u] = __ldg(xr + c0 + u * kWorkers);
                graw[u] = __ldg(gr + c0 + u * kWorkers);
            }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (c0 + u * kWorkers >= nv) continue;
            const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&raw[u]);
            const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&graw[u]);
            uint4 o;
            __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 f = __bfloat1622float2(b2[q]);
                const float2 g = __bfloat1622float2(g2[q]);
                o2[q] = __floats2bfloat162_rn(f.x * rs * g.x, f.y * rs * g.y);
            }
            outr[c0 + u * kWorkers] = o;
        }
    }
    worker_sync();  // the partials are read before a later row writes them
}

__global__ void __launch_bounds__(kThreads, 1)
mlp_chain_kernel(const __grid_constant__ CUtensorMap tm_wg, const __grid_constant__ CUtensorMap tm_wu,
                 const __grid_constant__ CUtensorMap tm_wd, const __grid_constant__ CUtensorMap tm_xhat,
                 const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_xhat64,
                 const __grid_constant__ CUtensorMap tm_h64, const __grid_constant__ MlpArgs p) {
    extern __shared__ uint8_t smem_raw[];
    const uint64_t t_start = globaltimer_ns();
    Ring ring;
    uint8_t* scratch;
    Ctl* ctl = cta_setup(smem_raw, 0, ring, &scratch);
    if (threadIdx.x == 0) trace_put(p.trace, p.trace_cap, 0, 2, 0, 0, t_start, globaltimer_ns());
    const WaitCtx wc{p.hdr, p.timeout_ns};
    const uint32_t tmem = ctl->tmem_base;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    MlpPlan P;
    P.B = p.B_host;
    if (p.d_B) P.B = *reinterpret_cast<const volatile int32_t*>(p.d_B);
    if (P.B < 0 || P.B > p.B_max) {
        if (blockIdx.x == 0 && threadIdx.x == 0) raise_error(wc, ET_ERR_BOUNDS, kWhereBoundsT);
        P.B = 0;
    }
    P.FT = p.F / kTileM;
    P.HT = p.H / kTileM;
    P.NR = ceil_div(P.B, kNormRows);
    P.MT = ceil_div(P.B, kWideNMax);
    // A CTA whose first task is a NORM runs it before anything else: its row
    // loads then reach memory ahead of the weight tiles every producer posts
    // (ahead of the norm's release) -- behind them a lone row's loads took
    // 7-9 us, and every gate/up tile waits for the norms.
    const bool early_norm = static_cast<int>(blockIdx.x) < P.NR;
    if (early_norm && warp >= kEpiWarp0) {
        norm_row(p, blockIdx.x, ctl);
        fence_proxy_async_global();  // x_hat is read by TMA
        worker_sync();
        if (threadIdx.x == kEpiWarp0 * 32) {
            __threadfence();
            red_release_add(&p.hdr->ev_norm, 1);
        }
    }
    // split of the down projection over F: the smallest divisor S of FT
    // (<= 16, chunks of >= 4 k-blocks) that gives every CTA a down tile, at
    // most 4 above 64 rows, whose fp32 partials (written, then read back,
    // 2 x B x H x 4 bytes a split) grow with the batch.  Measured on the
    // configured shape (H 4096, F 14336): S = 7 / 14 / 4 at B = 1 gave 89 /
    // 89 / 90 us, at B = 64 98 / 109 / 109 us; S = 4 against 7 at B = 128
    // 104 against 111 us, at B = 256 135 against 139 us.
    P.S = 1;
    if (P.MT > 0 && P.MT * P.HT < static_cast<int>(gridDim.x)) {
        const int cap = P.B > 64 ? 4 : kMlpSplitMax;
        for (int d = 2; d <= cap; ++d) {
            if (P.FT % d || p.F / d / kBlockK < 4) continue;
            P.S = d;
            if (P.MT * P.HT * d >= static_cast<int>(gridDim.x)) break;
        }
    }
    // K split of the gate/up tiles: with one row tile, F/128 tiles can leave
    // CTAs idle; the smallest split that gives the grid >= 2.5 tasks a CTA (K
    // chunks of >= 8 k-blocks, partial rows within gu_cap), else none
    P.KC = 1;
    {
        const int nkb = p.H / kBlockK, G = static_cast<int>(gridDim.x);
        for (int kc = 2; kc <= kGuSplitMax && P.MT * P.FT < (5 * G) / 2; kc *= 2) {
            if (nkb % kc || nkb / kc < 8 || P.B * kc > p.gu_cap) break;
            if (2 * P.MT * P.FT * kc >= 5 * G) {
                P.KC = kc;
                break;
            }
        }
    }
    P.n_gu = P.MT * P.FT * P.KC;
    P.n_dn = P.MT * P.S * P.HT;
    P.n_red = P.S > 1 ? ceil_div(P.B, kRedRows) * P.HT : 0;
    P.total = P.NR + P.n_gu + P.n_dn + P.n_red;

    auto gemm_of = [&](const MlpTile& t) {
        if (t.kind == 1) {
            const int nkb = p.H / kBlockK / P.KC;
            return GemmTask{&tm_wg, &tm_wu, &tm_xhat, p.b_wide ? &tm_xhat64 : nullptr,
                            t.ft * kTileM, t.mt * kWideNMax, t.kc * nkb, nkb, t.n,
                            &p.hdr->ev_norm, P.NR, kWhereNorm};
        }
        const int fchunk = p.F / P.S;
        return GemmTask{&tm_wd, nullptr, &tm_h, p.b_wide ? &tm_h64 : nullptr, t.ht * kTileM,
                        t.mt * kWideNMax, t.s * (fchunk / kBlockK), fchunk / kBlockK, t.n,
                        &p.ev_h[t.mt * kMlpSplitMax + t.s], P.FT / P.S, kWhereH};
    };

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first(), pol_b = policy_evict_last();
            int task = blockIdx.x;
            auto next = [&](GemmTask& g) {  // this CTA's next GEMM task
                for (; task < P.total; task += gridDim.x) {
                    const MlpTile t = mlp_tile(P, task);
                    if (t.kind == 1 || t.kind == 2) {
                        g = gemm_of(t);
                        task += gridDim.x;
                        return true;
                    }
                }
                return false;
            };
            produce_static(next, ring, ctl, wc, pol_w, pol_b);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            MmaState ms;
            for (int task = blockIdx.x; task < P.total; task += gridDim.x) {
                const MlpTile t = mlp_tile(P, task);
                if (t.kind == 0 || t.kind == 3) continue;
                auto ftr = [&](int u, uint64_t tp, uint64_t tl) {
                    trace_put(p.trace, p.trace_cap, t.kind == 1 ? kTaskGateUp : kTaskDown, 5, task,
                              u, tp, tl);
                };
                if (!mma_task(gemm_of(t), ring, ctl, ms, tmem, wc, ftr)) break;
            }
        }
        __syncwarp();
    } else if (warp >= kEpiWarp0) {
        const int q = warp & 3, half = (warp - kEpiWarp0) >> 2;  // TMEM lane quadrant, column half
        const int wtid = threadIdx.x - kEpiWarp0 * 32;
        const int H = p.H, F = p.F;
        EpiState es;
        for (int task = blockIdx.x + (early_norm ? gridDim.x : 0); task < P.total;
             task += gridDim.x) {
            const MlpTile t = mlp_tile(P, task);
            const uint64_t tw = p.trace ? globaltimer_ns() : 0;
            const int ttype = t.kind == 0 ? kTaskNorm : t.kind == 1 ? kTaskGateUp
                            : t.kind == 2 ? kTaskDown : kTaskReduce;
            TraceOnExit trace_task{p.trace, p.trace_cap, ttype, task, tw, wtid == 0};
            if (t.kind == 0) {
                norm_row(p, t.i, ctl);
                fence_proxy_async_global();
                worker_sync();
                if (wtid == 0) {
                    __threadfence();
                    red_release_add(&p.hdr->ev_norm, 1);
                }
                continue;
            }
            if (t.kind == 3) {  // REDUCE: row slice t.s of output column tile t.ht
                const int r0 = t.s * kRedRows, r1 = min(P.B, r0 + kRedRows);
                const int mt = r0 / kWideNMax;
                if (wtid == 0)
                    ctl->flag =
                        ev_wait_geq(wc, p.ev_y + mt * P.HT + t.ht, P.S, kWhereY) ? 1 : 0;
                worker_sync();
                if (!ctl->flag) break;
                reduce_slice4(p.partial, static_cast<size_t>(p.B_max) * H, H, P.S, r0, r1,
                              t.ht * kTileM, p.out, H);
                continue;
            }
            const bool two = t.kind == 1;
            uint32_t acc, acc1;
            if (!epi_acquire(ctl, es, two, t.n, tmem, wc, acc, acc1)) break;
            if (wtid == 0) trace_put(p.trace, p.trace_cap, ttype, 6, task, 0, tw, globaltimer_ns());
            const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
            const uint32_t lane_base = acc + lane_off;
            const size_t m0 = static_cast<size_t>(t.mt) * kWideNMax;
            if (t.kind == 1) {
                const int f = t.ft * kTileM + q * 32 + lane;
                // K-split tile: fp32 partials of chunk kc, rows of this call
                float* gpart = p.gu_part + (static_cast<size_t>(t.kc) * P.B) * F;
                float* upart = gpart + static_cast<size_t>(p.gu_cap) * F;
                for (int c0 = half * 16; c0 < t.n; c0 += 32) {
                    float gv[16], uv[16];
                    tmem_ld16(lane_base + c0, gv);
                    tmem_ld16(acc1 + lane_off + c0, uv);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        if (c0 + c >= t.rows) continue;
                        const size_t r = m0 + c0 + c;
                        if (P.KC == 1) {
                            p.h[r * F + f] =
                                __float2bfloat16_rn(gv[c] / (1.0f + __expf(-gv[c])) * uv[c]);
                        } else {
                            gpart[r * F + f] = gv[c];
                            upart[r * F + f] = uv[c];
                        }
                    }
                }
                epi_release(ctl, es, true, t.n);
                if (P.KC > 1) {  // the chunk that completes the tile sums the partials
                    int* ev = p.ev_gu + t.mt * P.FT + t.ft;
                    worker_sync();
                    if (wtid == 0) {
                        __threadfence();
                        ctl->flag = (atom_acq_rel_add(ev, 1) == P.KC - 1) ? 1 : 0;
                    }
                    worker_sync();
                    if (!ctl->flag) continue;
                    if (wtid == 0) *ev = 0;  // every chunk arrived: reset for the next call
                    const float* g0 = p.gu_part;
                    const float* u0 = p.gu_part + static_cast<size_t>(p.gu_cap) * F;
                    for (int j = wtid; j < t.rows * (kTileM / 4); j += kWorkers) {
                        const size_t r = m0 + j / (kTileM / 4);
                        const int ff = t.ft * kTileM + (j % (kTileM / 4)) * 4;
                        float gs[4] = {0.0f, 0.0f, 0.0f, 0.0f}, us[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                        for (int kc = 0; kc < P.KC; ++kc) {  // chunk order kc = 0 .. KC-1
                            const size_t o = (static_cast<size_t>(kc) * P.B + r) * F + ff;
                            const float4 gq = __ldcg(reinterpret_cast<const float4*>(g0 + o));
                            const float4 uq = __ldcg(reinterpret_cast<const float4*>(u0 + o));
                            gs[0] += gq.x; gs[1] += gq.y; gs[2] += gq.z; gs[3] += gq.w;
                            us[0] += uq.x; us[1] += uq.y; us[2] += uq.z; us[3] += uq.w;
                        }
                        __nv_bfloat162 o2[2];
#pragma unroll
                        for (int i2 = 0; i2 < 2; ++i2) {
                            const float a = gs[2 * i2], b2 = gs[2 * i2 + 1];
                            o2[i2] = __floats2bfloat162_rn(a / (1.0f + __expf(-a)) * us[2 * i2],
                                                           b2 / (1.0f + __expf(-b2)) * us[2 * i2 + 1]);
                        }
                        *reinterpret_cast<uint2*>(p.h + r * F + ff) = *reinterpret_cast<const uint2*>(o2);
                    }
                }
                fence_proxy_async_global();  // h is read back by TMA
                worker_sync();
                if (wtid == 0) {
                    const bool skip = p.fault_mode == 1 && t.mt * P.FT + t.ft == p.fault_arg;
                    __threadfence();
                    if (!skip) red_release_add(&p.ev_h[t.mt * kMlpSplitMax + t.ft / (P.FT / P.S)], 1);
                }
                continue;
            }
            // down projection tile
            const int hh = t.ht * kTileM + q * 32 + lane;
            for (int c0 = half * 16; c0 < t.n; c0 += 32) {
                float v[16];
                tmem_ld16(lane_base + c0, v);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    if (c0 + c >= t.rows) continue;
                    const size_t m = m0 + c0 + c;
                    if (P.S == 1)
                        p.out[m * H + hh] = __float2bfloat16_rn(v[c]);
                    else
                        p.partial[(static_cast<size_t>(t.s) * p.B_max + m) * H + hh] = v[c];
                }
            }
            epi_release(ctl, es, false, t.n);
            if (P.S > 1) {  // the partial is stored: count it on the tile's event
                worker_sync();
                if (wtid == 0) {
                    __threadfence();
                    red_release_add(p.ev_y + t.mt * P.HT + t.ht, 1);
                }
            }
        }
    }

    const uint64_t t_exit = globaltimer_ns();
    const bool aborted_run = ld_relaxed(&p.hdr->abort) != 0;
    cta_teardown(ctl, aborted_run);
    __syncthreads();
    if (threadIdx.x == 0) {
        trace_put(p.trace, p.trace_cap, 0, 3, 0, 0, t_exit, globaltimer_ns());
        __threadfence();
        ctl->flag = (atomicAdd(&p.hdr->exit_count, 1) == static_cast<int>(gridDim.x) - 1) ? 1 : 0;
    }
    __syncthreads();
    if (ctl->flag) {
        __threadfence();
        const bool ab = ld_relaxed(&p.hdr->abort) != 0;
        const int mt_clear = ab ? p.mt_max : P.MT;
        for (int j = threadIdx.x; j < mt_clear * kMlpSplitMax; j += kThreads) p.ev_h[j] = 0;
        const int y_clear = ab ? p.mt_max : (P.S > 1 ? P.MT : 0);
        for (int j = threadIdx.x; j < y_clear * P.HT; j += kThreads) p.ev_y[j] = 0;
        if (ab)  // the K-split counters reset themselves unless the launch aborted
            for (int j = threadIdx.x; j < p.mt_max * P.FT; j += kThreads) p.ev_gu[j] = 0;
        __syncthreads();
        if (threadIdx.x == 0) {
            p.hdr->ev_norm = 0;
            p.hdr->abort = 0;
            __threadfence();
            p.hdr->exit_count = 0;
        }
    }
}

int mlp_smem_bytes() { return smem_bytes_for(0); }

cudaError_t launch_mlp(const MlpArgs& a, const CUtensorMap* maps, int grid, int smem,
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
    return cudaLaunchKernelEx(&cfg, mlp_chain_kernel, maps[0], maps[1], maps[2], maps[3], maps[4],
                              maps[5], maps[6], a);
}

cudaError_t prepare_mlp(int smem) {
    return cudaFuncSetAttribute(mlp_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem);
}

}  // namespace et
