// splitk_kernel.cu -- split-K GEMM whose partial sums meet through event
// counters instead of a second kernel:
//   Y[M,N] = bf16( sum_{s < split} X[:, K_s] Wt[:, K_s]^T )
// Task (mt, nt, s) computes an fp32 partial of a 256 x 128 output tile over
// K chunk s and adds 1 to the tile's counter with acquire-release order; the
// task that sees split-1 sums the partials in chunk order, stores Y and puts
// the counter back to zero.  No task waits, so the schedule cannot deadlock.
// M stays symbolic: it may be read from device memory, and the same compiled
// kernel serves every M up to M_max.
//
// Source: "Prompt Boundary-Aware Scheduling with Event Tensors for Dynamic
// Kernels" -- the split-K summation example, where the reduction is gated by
// an event over the producing tiles rather than by a kernel boundary.
#include "et_gemm.cuh"

namespace et {

__global__ void __launch_bounds__(kThreads, 1)
splitk_kernel(const __grid_constant__ SplitKArgs p, const __grid_constant__ CUtensorMap tm_w,
              const __grid_constant__ CUtensorMap tm_x) {
    extern __shared__ uint8_t smem_raw[];
    Ring ring;
    Ctl* ctl = cta_setup(smem_raw, p.stages, kWideNMax, ring);
    const WaitCtx wc{p.hdr, p.timeout_ns};
    const uint32_t tmem = ctl->tmem_base;
    Pipe pipe;

    int M = p.d_M ? *reinterpret_cast<const volatile int32_t*>(p.d_M) : p.M_host;
    if (M < 0 || M > p.M_max) {
        if (blockIdx.x == 0 && threadIdx.x == 0) raise_error(wc, ET_ERR_BOUNDS, kWhereBoundsT);
        M = 0;
    }
    if (threadIdx.x == 0) {
        tma_prefetch_map(&tm_w);
        tma_prefetch_map(&tm_x);
    }
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_b = policy_evict_last();
    const int N = p.N, split = p.split;
    const int MT = ceil_div(M, kWideNMax), NT = N / kTileM;
    const int kbs = p.K / kBlockK / split;
    const int total = MT * NT * split;

    bool ok = true;
    for (int task = blockIdx.x; task < total; task += gridDim.x) {
        if (threadIdx.x == 0) ctl->fail = 0;
        __syncthreads();
        const int s = task % split, rest = task / split;
        const int nt = rest % NT, mt = rest / NT;
        const int rows = min(kWideNMax, M - mt * kWideNMax);
        const int n = (rows + 15) / 16 * 16;
        GemmTask t{&tm_w, nullptr, &tm_x, nt * kTileM, mt * kWideNMax, s * kbs, kbs, n,
                   n <= kWideNMax / 2 ? 2 : 1, nullptr, 0, 0};
        bf16* Y = p.Y;
        float* part = p.partial;
        const int m0 = mt * kWideNMax, Mmax = p.M_max;
        ok = run_gemm_task(t, ctl, ring, pipe, tmem, wc, pol_w, pol_b, [&](int q, int ln) {
            const int col = nt * kTileM + q * 32 + ln;
            const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
            for (int c0 = 0; c0 < n; c0 += 16) {
                float v[16];
                tmem_ld16(lane_base + c0, v);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    if (c0 + c >= rows) continue;
                    const size_t m = static_cast<size_t>(m0 + c0 + c);
                    if (split == 1)
                        Y[m * N + col] = __float2bfloat16_rn(v[c]);
                    else
                        part[(static_cast<size_t>(s) * Mmax + m) * N + col] = v[c];
                }
            }
        });
        if (!ok) break;
        if (split > 1) {
            int* ev = p.ev + mt * NT + nt;
            if (threadIdx.x == 0) {
                __threadfence();
                ctl->flag = (atom_acq_rel_add(ev, 1) == split - 1) ? 1 : 0;
            }
            __syncthreads();
            if (ctl->flag) {
                for (int i = threadIdx.x; i < rows * kTileM; i += kThreads) {
                    const size_t m = static_cast<size_t>(m0 + i / kTileM);
                    const int col = nt * kTileM + (i % kTileM);
                    float sum = 0.0f;
                    for (int s2 = 0; s2 < split; ++s2)
                        sum += __ldcg(part + (static_cast<size_t>(s2) * Mmax + m) * N + col);
                    Y[m * N + col] = __float2bfloat16_rn(sum);
                }
                if (threadIdx.x == 0) *ev = 0;  // every split has arrived: reset for the next call
            }
            __syncthreads();
        }
    }
    if (!ok) drain_after_failure(ctl, ring, pipe);
    cta_teardown(ctl);
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
    return cudaLaunchKernelEx(&cfg, splitk_kernel, a, maps[0], maps[1]);
}

cudaError_t prepare_splitk(int smem) {
    return cudaFuncSetAttribute(splitk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

}  // namespace et
