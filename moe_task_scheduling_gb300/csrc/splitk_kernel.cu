// splitk_kernel.cu -- split-K GEMM whose partial sums meet through event
// counters instead of a second kernel:
//   Y[M,N] = bf16( sum_{s < split} X[:, K_s] Wt[:, K_s]^T )
// Static schedule (task t runs on CTA t mod grid; every role walks the same
// task list):
//   [0, G)        TILE (mt, nt, s): fp32 partial of a 256 x 128 output tile over
//                 K chunk s (bf16 Y directly when split == 1); releases
//                 ev[mt][nt]
//   [G, G + R)    REDUCE (q, nt), split > 1 only: waits ev[tile] >= split, then
//                 sums rows [32q, 32q + 32) of the tile's partials in chunk
//                 order and stores bf16 Y.
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
    constexpr int kRedRows = 32;  // rows per reduce task
    const int n_red = split > 1 ? ceil_div(M, kRedRows) * NT : 0;

    auto gemm_of = [&](const SplitKTile& t) {
        return GemmTask{&tm_w, nullptr, &tm_x, p.b_wide ? &tm_x64 : nullptr, t.nt * kTileM,
                        t.mt * kWideNMax, t.s * kbs, kbs, t.n, t.nt, nullptr, 0, 0};
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
        const int q = warp & 3, half = (warp - kEpiWarp0) >> 2;  // TMEM lane quadrant, column half
        const int wtid = threadIdx.x - kEpiWarp0 * 32;
        EpiState es;
        for (int task = blockIdx.x; task < total + n_red; task += gridDim.x) {
            if (task >= total) {  // REDUCE: row slice qs of tile column nt
                const int r = task - total, nt = r % NT, qs = r / NT;
                const int r0 = qs * kRedRows, r1 = min(M, r0 + kRedRows), mt = r0 / kWideNMax;
                if (wtid == 0)
                    ctl->flag = ev_wait_geq(wc, p.ev + mt * NT + nt, split, kWhereY) ? 1 : 0;
                worker_sync();
                if (!ctl->flag) break;
                reduce_slice(p.partial, static_cast<size_t>(p.M_max) * N, N, split, r0, r1,
                             nt * kTileM, p.Y, N);
                continue;
            }
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
            if (split > 1) {  // the partial is stored: count it on the tile's event
                worker_sync();
                if (wtid == 0) {
                    __threadfence();
                    red_release_add(p.ev + t.mt * NT + t.nt, 1);
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

int splitk_smem_bytes() { return smem_bytes_for(0); }

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
