// splitk_kernel.cu -- split-K GEMM whose partial sums meet through event
// counters instead of a second kernel:
//   Y[M,N] = bf16( sum_{s < split} X[:, K_s] Wt[:, K_s]^T )
// Task (mt, nt, s) computes an fp32 partial of a 256 x 128 output tile over
// K chunk s and adds 1 to the tile's counter with acquire-release order; the
// task that sees split-1 sums the partials in chunk order, stores Y and puts
// the counter back to zero.  No task waits on another, so the schedule cannot
// deadlock.  M stays symbolic: it may be read from device memory, and the same
// compiled kernel serves every M up to M_max.
//
// Schedule: static, task t runs on CTA t mod grid; every role walks the same
// task list.
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
              const __grid_constant__ SplitKArgs p) {
    extern __shared__ uint8_t smem_raw[];
    Ring ring;
    uint8_t* scratch;
    Ctl* ctl = cta_setup(smem_raw, 0, ring, &scratch);
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

    auto gemm_of = [&](const SplitKTile& t) {
        return GemmTask{&tm_w, nullptr, &tm_x, t.nt * kTileM, t.mt * kWideNMax, t.s * kbs, kbs,
                        t.n, nullptr, 0, 0};
    };

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first(), pol_b = policy_evict_last();
            ProdState ps;
            for (int task = blockIdx.x; task < total; task += gridDim.x)
                if (!produce_task(gemm_of(splitk_tile(task, split, NT, M)), ring, ctl, ps, wc, pol_w,
                                  pol_b))
                    break;
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            MmaState ms;
            for (int task = blockIdx.x; task < total; task += gridDim.x)
                if (!mma_task(gemm_of(splitk_tile(task, split, NT, M)), ring, ctl, ms, tmem, wc))
                    break;
        }
        __syncwarp();
    } else if (warp >= kEpiWarp0) {
        const int q = warp - kEpiWarp0, wtid = threadIdx.x - kEpiWarp0 * 32;
        EpiState es;
        for (int task = blockIdx.x; task < total; task += gridDim.x) {
            const SplitKTile t = splitk_tile(task, split, NT, M);
            uint32_t acc, acc1;
            if (!epi_acquire(ctl, es, false, t.n, tmem, wc, acc, acc1)) break;
            const int col = t.nt * kTileM + q * 32 + lane;
            const uint32_t lane_base = acc + (static_cast<uint32_t>(q * 32) << 16);
            const size_t m0 = static_cast<size_t>(t.mt) * kWideNMax;
            for (int c0 = 0; c0 < t.n; c0 += 16) {
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
            if (split > 1) {
                int* ev = p.ev + t.mt * NT + t.nt;
                worker_sync();  // every partial of this CTA is stored
                if (wtid == 0) {
                    __threadfence();
                    ctl->flag = (atom_acq_rel_add(ev, 1) == split - 1) ? 1 : 0;
                }
                worker_sync();
                if (ctl->flag) {  // last arriver: sum the partials in split order
                    for (int i = wtid; i < t.rows * kTileM; i += kWorkers) {
                        const size_t m = m0 + i / kTileM;
                        const int cc = t.nt * kTileM + (i % kTileM);
                        float sum = 0.0f;
                        for (int s2 = 0; s2 < split; ++s2)
                            sum += __ldcg(p.partial + (static_cast<size_t>(s2) * p.M_max + m) * N + cc);
                        p.Y[m * N + cc] = __float2bfloat16_rn(sum);
                    }
                    if (wtid == 0) *ev = 0;  // every split has arrived: reset for the next call
                }
            }
        }
    }

    const bool aborted_run = ld_relaxed(&p.hdr->abort) != 0;
    cta_teardown(ctl, aborted_run);
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(&p.hdr->exit_count, 1) == static_cast<int>(gridDim.x) - 1) {
            // an aborted launch may leave tile counters behind: clear them all
            if (ld_relaxed(&p.hdr->abort) != 0) {
                const int n_ev = ceil_div(p.M_max, kWideNMax) * (N / kTileM);
                for (int i = 0; i < n_ev; ++i) p.ev[i] = 0;
                p.hdr->abort = 0;
            }
            __threadfence();
            p.hdr->exit_count = 0;
        }
    }
}

int splitk_smem_bytes() { return smem_bytes_for(0); }

cudaError_t launch_splitk(const SplitKArgs& a, const CUtensorMap* maps, int grid, int smem,
                          cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, splitk_kernel, maps[0], maps[1], a);
}

cudaError_t prepare_splitk(int smem) {
    return cudaFuncSetAttribute(splitk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

}  // namespace et
