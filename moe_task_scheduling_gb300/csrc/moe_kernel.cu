// moe_kernel.cu -- the MoE layer as one persistent megakernel whose tiled
// tasks are ordered by device-resident event counters, not kernel boundaries.
//
// Task graph (one task index space, claimed with an atomic head by each
// CTA's producer thread and handed to its MMA thread and worker warps through
// a small shared-memory ring; index order is a topological order and every
// role of a CTA walks its tasks in that order, so every wait is on a task
// that a resident CTA already holds -- the launch is cooperative):
//   [0, R*C)    ROUTER r,c fixed-order fp32 logits of router tile r for expert
//                          chunk c; the chunk that completes the tile (counter
//                          ev_tile[r]) takes the top-k, gate weights and the
//                          tile's expert histogram; the tile that completes
//                          ev_router (count R, computed from the device token
//                          count; a single tile is its own last) runs the
//                          SCAN: counts, offsets, the expert row tiles, the
//                          splits and the down-tile width, which it publishes
//                          -- the queue below is implicit, each producer
//                          decodes the index it claims -- and, with a single
//                          router tile, it then writes the permutation indices
//                          (no row moves: that batch's gate/up tiles read the
//                          tile's token rows in place):
//   queue:      PERMUTE r,q stable scatter of part q of router tile r's rows;
//                          releases ev_perm
//               GATEUP g,f SwiGLU tile of expert row-tile g, F-tile f (waits
//                          ev_perm >= permute parts); releases ev_h[g][chunk(f)]
//               DOWN g,s,n down-projection tile (128 output columns, or 256
//                          for tall row tiles), F-chunk s (waits ev_h[g][s] >=
//                          F-tiles per chunk); with a split the last arriver on
//                          ev_y[g][n] sums the fp32 partials in chunk order;
//                          a finished output tile adds to ev_gdone[g]
//               COMBINE c  waits for ev_gdone of every row tile that holds one
//                          of its tokens' rows, out = sum_j w * y; a single
//                          combine is run inline by the output tile that
//                          completes ev_ydone.
//
// Sources: "Prompt Boundary-Aware Scheduling with Event Tensors for Dynamic
// Kernels" (MoE routing gives data-dependent event counters that trigger
// tasks; split-K partials summed through events; symbolic batch size) and
// "Megakernels ch. 5 - Event Tensor et le dynamisme" section 5.5 (targets
// computed on the GPU before waiting; online balancing with atomics).
#include <cstring>

#include "et_gemm.cuh"

namespace et {

// One layer's tensor maps: its weights and its staging buffers (gate, up,
// down; permuted x and h in 16- and 64-row boxes; router weight; the fused
// block's shared expert, x_hat and shared h; the rows the router reads -- x,
// or x_hat in a fused block -- in 16-row boxes, the gate/up activations of a
// batch of one router tile).
struct MoeLayerMaps {
    CUtensorMap wg, wu, wd, xp, h, wr, xp64, h64, sg, su, sd, xn, hs, xr;
};
constexpr int kMapsPerLayer = 14;

// The kernel parameter: nl <= kN chained layers; layer l + 1 reads layer l's
// output.  A single layer launches with kN = 1: a 2 KB parameter block instead
// of 8 KB (measured on GB300: about 1 us less launch latency).
template <int kN>
struct MoeLaunch {
    MoeLayerMaps m[kN];
    MoeArgs a[kN];
    int nl;
};
template <bool kChain>
using MoeLaunchOf = MoeLaunch<kChain ? kMaxLayers : 1>;

__device__ __forceinline__ int layer_of(const TaskMsg& m) { return (m.type >> kLayerShift) & 3; }

__device__ __forceinline__ void unpack8(const uint4& raw, float (&v)[8]) {
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(b2[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}

__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
    uint4 raw;
    __nv_bfloat162* b2 = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) b2[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    return raw;
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + __expf(-g)) * u; }

__device__ __forceinline__ int wtid_() { return static_cast<int>(threadIdx.x) - kEpiWarp0 * 32; }

// SIMT scratch (bytes): router logits [16][256] f32 at 0, the tile's expert
// histogram at kHistOff, its top-k picks at kSelOff; the scan's arrays at 0
// (after the logits are dead); permute rows at kPermOff.
constexpr int kMoeScratch = 18432;
constexpr int kHistOff = kRouterTile * 256 * 4;  // int [256]
constexpr int kSelOff = kHistOff + 256 * 4;      // int [16 * 8]
constexpr int kPermOff = 8192;                   // int [128] entries, int [128] rows
constexpr int kPlanOff = kSelOff + 512;          // MoePlan [kMaxLayers], set once per launch

// Speculative L2 prefetch of a producer's predicted first gate/up tile while
// routing runs (see spec_prefetch): KB of weights a producer (measured on the
// Mixtral shape: +0.7 % over the sweep with 512 or 1024, T >= 16 gaining).
constexpr int kSpecPrefetchKb = 512;

// ------------------------------------------------------------------ trace

// Optional per-task record (see et_opts.trace): {type | role << 8, a, b, cta,
// t_begin, t_end}.  role 0 = producer (pop .. loads issued), 1 = workers
// (task received .. done), 2 = CTA (start .. set-up done), 3 = CTA exit,
// 5 = MMA issuer, one per fill (posted .. its bytes landed; b = fill index),
// 6 = workers (GEMM task received .. its accumulator ready).
__device__ __forceinline__ void trace_rec(const MoeArgs& p, int type, int role, int a, int b,
                                          uint64_t t0, uint64_t t1) {
    trace_put(p.trace, p.trace_cap, type, role, a, b, t0, t1);
}

// Sub-phase marks of the front end (worker thread 0, role 4): type 16 + id
// spans [t_prev, now]; returns now.
__device__ __forceinline__ uint64_t phase_mark(const MoeArgs& p, int id, uint64_t t_prev) {
    if (!p.trace || wtid_() != 0) return t_prev;
    __shared__ long long c_prev;  // SM cycles at the previous mark (field a: cycles in the phase)
    const long long c = clock64();
    const uint64_t t = globaltimer_ns();
    trace_rec(p, 16 + id, 4, static_cast<int>(c - c_prev), 0, t_prev, t);
    c_prev = clock64();
    return globaltimer_ns();
}

struct TraceScope {  // records the workers' task on scope exit (worker thread 0)
    const MoeArgs& p;
    int type, a, b;
    uint64_t t0;
    bool on;
    __device__ __forceinline__ ~TraceScope() {
        if (on) trace_rec(p, type, 1, a, b, t0, globaltimer_ns());
    }
};

// ------------------------------------------------------------------ ROUTER

// Fixed-order logits of nt (<= 16) tokens x `ec` experts (global experts
// e0 .. e0+ec).  A job is TB tokens x EBW experts on one warp: lane l owns
// partial sum l and accumulates h = l, l+32, ... in ascending order with fp32
// fma (a bf16 x bf16 product is exact in fp32, so fma == mul + add); the
// halving shuffle tree (16, 8, 4, 2, 1) then adds p[l] + p[l + off].
// Token rows: xb + t * H.  Weight element (h, j) of chunk column j sits at
//   wb + ((o + j) >> 3) * blk + h * rs + ((o + j) & 7)
// which covers the [H, E] layout in global memory (o = 0, blk = 8, rs = E)
// and the staged one (blocks of 8 experts, 16 bytes a row).  EBW divides
// both ec and 8, so a job's EBW columns never straddle a block.  Logit
// (t, e0 + j) goes to out[t * E + e0 + j].
// Weights of EBW experts at one h (shared-window address `sa`) as bf16 bit
// patterns.
template <int EBW>
__device__ __forceinline__ void load_w16(uint32_t sa, uint16_t (&w)[EBW]) {
    uint32_t u[(EBW + 1) / 2];
    if constexpr (EBW == 8) {
        const uint4 v = lds_v4(sa);
        u[0] = v.x, u[1] = v.y, u[2] = v.z, u[3] = v.w;
    } else if constexpr (EBW == 4) {
        const uint2 v = lds_v2(sa);
        u[0] = v.x, u[1] = v.y;
    } else if constexpr (EBW == 2) {
        u[0] = lds_u32(sa);
    } else {
        u[0] = lds_u16(sa);
    }
#pragma unroll
    for (int b = 0; b < EBW; ++b)
        w[b] = static_cast<uint16_t>((b & 1) ? (u[b >> 1] >> 16) : (u[b >> 1] & 0xffffu));
}

template <int EBW, int TB>
__device__ __forceinline__ void router_logits_body(const MoeArgs& p, const bf16* xb,
                                                   const bf16* wb, int o, int rs, int blk, int nt,
                                                   int e0, int ec, float* out) {
    const int H = p.H, E = p.E;
    const int warp = wtid_() >> 5, lane = wtid_() & 31;
    const int neb = ec / EBW, ntb = ceil_div(nt, TB);
    for (int job = warp; job < neb * ntb; job += kWorkers / 32) {
        const int tb = job / neb, j0 = (job % neb) * EBW;
        const int tn = min(TB, nt - tb * TB);
        float acc[TB][EBW];
#pragma unroll
        for (int a = 0; a < TB; ++a)
#pragma unroll
            for (int b = 0; b < EBW; ++b) acc[a][b] = 0.0f;
        // rows past the tile's last token repeat that token (in bounds; their
        // sums are never stored)
        int xrow[TB];
#pragma unroll
        for (int a = 0; a < TB; ++a) xrow[a] = (tb * TB + min(a, tn - 1)) * H;
        const bf16* wj = wb + static_cast<size_t>((o + j0) >> 3) * blk + ((o + j0) & 7);
        const uint32_t xs = smem_u32(xb), ws = smem_u32(wj);
        // One fp32 fma with bf16 operands (fma.rn.f32.bf16) per product: the
        // operands need no widening moves.  Measured in isolation on GB300, a
        // 16-token x 32-expert tile over H = 2048 on 8 warps: 15.0K SM cycles,
        // against 18.6K for packed fp32x2 fmas fed by bf16 -> fp32 unpacking,
        // and 24.4K for the latter through generic pointers into shared memory
        // (hence the shared-window loads).  Unrolled twice: this code often
        // runs once per call, cold after the flush.
#pragma unroll 2
        for (int h = lane; h < H; h += 32) {  // h ascending per lane
            uint16_t wv[EBW];
            load_w16<EBW>(ws + static_cast<uint32_t>(h * rs) * 2u, wv);
            uint16_t xv[TB];
#pragma unroll
            for (int a = 0; a < TB; ++a) xv[a] = lds_u16(xs + static_cast<uint32_t>(xrow[a] + h) * 2u);
#pragma unroll
            for (int a = 0; a < TB; ++a)
#pragma unroll
                for (int b = 0; b < EBW; ++b) acc[a][b] = fma_bf16(xv[a], wv[b], acc[a][b]);
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1)
#pragma unroll
            for (int a = 0; a < TB; ++a)
#pragma unroll
                for (int b = 0; b < EBW; ++b)
                    acc[a][b] = acc[a][b] + __shfl_down_sync(0xffffffffu, acc[a][b], off);
        // Lane i (< TB * EBW) takes logit (i / EBW, i % EBW) from lane 0, where
        // the halving tree left every sum, and stores it with its bias: one
        // load and one store for the job.  (Lane 0 storing them one by one
        // took ~2.7K SM cycles a 4 x 8 job: each bias load waited for the
        // previous logit's store, as the two arrays may alias.)
        float v = 0.0f;
#pragma unroll
        for (int a = 0; a < TB; ++a)
#pragma unroll
            for (int b = 0; b < EBW; ++b) {
                const float sum = __shfl_sync(0xffffffffu, acc[a][b], 0);
                if (lane == a * EBW + b) v = sum;
            }
        const int la = lane / EBW, lb = lane % EBW;
        if (lane < TB * EBW && la < tn) {
            float L = v;
            if (p.bias) L = L + p.bias[e0 + j0 + lb];
            out[(tb * TB + la) * E + e0 + j0 + lb] = L;
        }
    }
}

// Tiles read in place (the router weight could not be staged): the same
// order through generic pointers, one (token, expert) logit a warp at a time
// (a fallback for expert counts without 8-expert weight blocks).
static __device__ __noinline__ void router_logits_inplace(int H, int E, const float* bias,
                                                          const bf16* xb, const bf16* wb, int o,
                                                          int rs, int blk, int nt, int e0, int ec,
                                                          float* out) {
    const int warp = wtid_() >> 5, lane = wtid_() & 31;
    for (int job = warp; job < nt * ec; job += kWorkers / 32) {
        const int t = job / ec, j = job % ec;
        const bf16* xr = xb + static_cast<size_t>(t) * H;
        const bf16* wj = wb + static_cast<size_t>((o + j) >> 3) * blk + ((o + j) & 7);
        float acc = 0.0f;
        for (int h = lane; h < H; h += 32)
            acc = fmaf(bf2f(xr[h]), bf2f(wj[static_cast<size_t>(h) * rs]), acc);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) acc = acc + __shfl_down_sync(0xffffffffu, acc, off);
        if (lane == 0) out[t * E + e0 + j] = bias ? acc + bias[e0 + j] : acc;
    }
}

// Narrow staged jobs (up to 16 accumulators) run out of line, so their
// registers do not add to the kernel's; the 4x8 job (many to a CTA on large
// batches) stays inline, which measured faster there.
template <int EBW, int TB>
static __device__ __noinline__ void router_logits_narrow(const MoeArgs& p, const bf16* xb,
                                                         const bf16* wb, int o, int rs, int blk,
                                                         int nt, int e0, int ec, float* out) {
    router_logits_body<EBW, TB>(p, xb, wb, o, rs, blk, nt, e0, ec, out);
}
template <int EBW, int TB>
__device__ __forceinline__ void router_logits(const MoeArgs& p, const bf16* xb, const bf16* wb,
                                              int o, int rs, int blk, int nt, int e0, int ec,
                                              float* out) {
    if constexpr (TB * EBW >= 32)
        router_logits_body<EBW, TB>(p, xb, wb, o, rs, blk, nt, e0, ec, out);
    else
        router_logits_narrow<EBW, TB>(p, xb, wb, o, rs, blk, nt, e0, ec, out);
}

// Router-weight staging geometry: 8-expert column blocks, rows padded to the
// TMA box height.
__device__ __forceinline__ int wr_rows_pad(int H, int box) { return (H + box - 1) / box * box; }

// 8-expert blocks a chunk of ec experts spans (0: the chunk cannot be staged).
__device__ __forceinline__ int wr_blocks(int ec) {
    return ec % 8 == 0 ? ec / 8 : (8 % ec == 0 ? 1 : 0);
}

// The per-call plan: a pure function of the device token count, the shapes
// and the grid, so every CTA and every role derives the same task numbering.
struct MoePlan {
    int T, R;      // tokens; router tiles of kRouterTile tokens
    int C, EC;     // router expert chunks per tile, experts per chunk
    int Q;         // permute parts per router tile
    int CT, NC;    // tokens per combine task; combine tasks
    int NP;        // permute tasks in the queue (0: one router tile, permuted inline)
    int NPW;       // permute releases the gate/up tiles wait for (the inline permute: 1)
    bool stage;    // router tiles stage x and their weight chunk in the ring
    bool wr_whole; // ... the whole router weight [H, E] with one bulk copy, as laid out
    // fused block: norm tasks (16 rows each; none when the router tiles stage
    // and normalise their rows), shared expert row tiles (256 rows), F-tiles and
    // down split; the static prefix [norm][router][shared gate/up] precedes the
    // routing-driven queue, which holds the shared down tiles
    int NRN, MTS, FTS, SS, NSG, NSD, NS0;
    bool spec;     // idle producers prefetch their predicted first gate/up tile (see pop_task)
};
static_assert(kPlanOff + kMaxLayers * sizeof(MoePlan) <= kMoeScratch, "plans fit the scratch");

__device__ __forceinline__ MoePlan moe_plan(const MoeArgs& p, int T, int G, uint32_t ring_bytes) {
    const int E = p.E, k = p.k, H = p.H;
    MoePlan P;
    P.T = T;
    P.R = ceil_div(T, kRouterTile);
    // Split the router's experts into chunks when there are few router tiles,
    // so a small batch still spreads over many CTAs; a chunk keeps at least two
    // experts (or all of E).
    const int want = P.R > 0 ? max(1, G / P.R) : 1;
    const int ecmin = min(E, 2);
    P.C = 1;  // chunk counts are powers of two (a cheap, uniform search)
    for (int d = 2; d <= E; d <<= 1)
        if (E % d == 0 && d <= want && E / d >= ecmin) P.C = d;
    // Staging: the smallest chunking (at least the one above) whose weight
    // blocks fit in the ring next to a full token tile.
    P.stage = false;
    if (p.wr_box > 0) {
        const uint32_t xpad = (static_cast<uint32_t>(min(T, kRouterTile) * H * 2) + 1023u) & ~1023u;
        const uint32_t hp = static_cast<uint32_t>(wr_rows_pad(H, p.wr_box));
        const uint32_t gb = p.gamma ? static_cast<uint32_t>(H) * 2u : 0u;  // gamma, fused norm
        for (int d = P.C; d <= E && !P.stage; d <<= 1) {
            if (E % d) break;
            const int nb = wr_blocks(E / d);
            if (nb > 0 && xpad + static_cast<uint32_t>(nb) * hp * 16u + gb <= ring_bytes) {
                P.C = d;
                P.stage = true;
            }
        }
    }
    P.EC = E / P.C;
    // A router weight small enough to sit next to a full token tile is staged
    // whole by one bulk copy (and reused by every later router task of the
    // CTA): 16-byte-wide TMA boxes of an 8-expert block move its rows far
    // below the bulk copy's rate.
    {
        const uint32_t xpad = (static_cast<uint32_t>(min(T, kRouterTile) * H * 2) + 1023u) & ~1023u;
        const uint32_t gb = p.gamma ? static_cast<uint32_t>(H) * 2u : 0u;
        const uint32_t wfull = static_cast<uint32_t>(H) * static_cast<uint32_t>(E) * 2u;
        P.wr_whole = P.stage && wfull % 16u == 0 &&
                     (reinterpret_cast<uintptr_t>(p.wr) & 15u) == 0 &&
                     xpad + wfull + gb <= ring_bytes;
    }
    P.Q = P.R > 0 ? min(max(1, G / P.R), kRouterTile * k) : 1;
    // a combine task's k rows per token fit the ring in one staging batch
    const int rpt = k + (p.gamma ? 1 : 0) + (p.gamma && p.Fs > 0 ? 1 : 0);  // rows per token
    const int per_batch = max(1, static_cast<int>(ring_bytes / (static_cast<uint32_t>(rpt) * H * 2)));
    P.CT = min(min(kCombineTile, per_batch), max(1, ceil_div(T, G)));
    P.NC = ceil_div(T, P.CT);
    P.NP = P.R > 1 ? P.R * P.Q : 0;
    P.NPW = P.R > 1 ? P.NP : 1;
    const int HT = H / kTileM;
    const bool block = p.gamma != nullptr;
    // a staged router tile normalises its own rows; otherwise NORM tasks do
    P.NRN = (block && !P.stage) ? P.R : 0;
    P.MTS = (block && p.Fs > 0) ? ceil_div(T, kWideNMax) : 0;
    P.FTS = p.Fs / kTileM;
    // the shared down tiles run beside the routed ones: split over F only for
    // small batches (short tiles, cheap reductions), to about half a task a CTA
    P.SS = 1;
    if (P.MTS > 0 && T <= 128 && T <= p.split_rows_cap && 2 * P.MTS * HT < G) {
        for (int d = 2; d <= kSplitMax; ++d) {
            if (P.FTS % d) continue;
            if (p.Fs / kBlockK / d < 4) break;  // keep >= 4 k-blocks a chunk
            P.SS = d;
            if (2 * P.MTS * HT * d >= G) break;
        }
    }
    P.NSG = P.MTS * P.FTS;
    P.NSD = P.MTS * P.SS * HT;
    P.NS0 = P.NRN + P.R * P.C + P.NSG;  // shared down tiles are queued by the scan
    // With few experts and many tokens every expert is active (each expects
    // >= 4 rows; one row tile an expert up to 256 rows) and there are enough
    // gate/up tiles that they are not split along K, so the queue's first
    // gate/up tasks are known before routing: expert 0's F-tiles in order, then
    // expert 1's ... (see queue_task).
    const int FTp = p.F / kTileM;
    P.spec = kSpecPrefetchKb > 0 && E <= 16 && T * k >= 4 * E && T * k <= kMoeNMax * E &&
             E * FTp >= 3 * G && !p.gamma && !p.ev_in;
    return P;
}

__device__ __forceinline__ bool scan_task(const MoeArgs& p, const MoePlan& P, uint8_t* smem,
                                          const Ring& ring, Ctl* ctl, const WaitCtx& wc,
                                          uint32_t& sphase, uint32_t& seq);

// ------------------------------------------------------------------ chained layers

// This layer's input rows of router tile r are the previous layer's output:
// wait (worker thread 0, bounded) until that layer's combine has released
// them.  Every worker then fences, so the rows can be read by bulk copies.
__device__ __forceinline__ bool wait_input(const MoeArgs& p, const MoePlan& P, int r, Ctl* ctl,
                                           const WaitCtx& wc) {
    if (!p.ev_in) return true;
    if (wtid_() == 0)
        ctl->flag = ev_wait_geq(wc, p.ev_in + r, min(kRouterTile, P.T - r * kRouterTile),
                                kWhereInput) ? 1 : 0;
    worker_sync();
    const bool ok = ctl->flag != 0;
    fence_proxy_async_global();
    worker_sync();  // the flag is read before any later task writes it
    return ok;
}

// Output rows [t0, t0 + nt) are stored: release them to the next layer, one
// count per row, on the counter of each 16-token tile they fall in.
__device__ __forceinline__ void release_output(const MoeArgs& p, int t0, int nt) {
    if (!p.ev_tok || nt <= 0) return;
    fence_proxy_async_global();  // read back by bulk copies in the next layer
    worker_sync();
    if (wtid_() == 0) {
        __threadfence();
        for (int r = t0 / kRouterTile; r * kRouterTile < t0 + nt; ++r) {
            const int lo = max(t0, r * kRouterTile), hi = min(t0 + nt, (r + 1) * kRouterTile);
            red_release_add(p.ev_tok + r, hi - lo);
        }
    }
}

// ------------------------------------------------------------------ NORM (fused block)

// x_hat rows of router tile r, defined in fp32 so the routing that depends on
// them is reproducible bit for bit: the sum of squares in the router-logit
// order (lane l sums h = l, l + 32, ... -- each square exact in fp32 -- then
// the halving tree), r = 1 / sqrt(ss / H + eps), x_hat = bf16((x * r) * gamma),
// every step one IEEE-rounded fp32 operation.  Warp w takes rows 2w, 2w + 1.
__device__ __forceinline__ void norm_task(const MoeArgs& p, const MoePlan& P, int r) {
    const int H = p.H, warp = wtid_() >> 5, lane = wtid_() & 31;
    constexpr int kRowsPerWarp = kRouterTile / (kWorkers / 32);
    for (int q = 0; q < kRowsPerWarp; ++q) {
        const int t = r * kRouterTile + warp * kRowsPerWarp + q;
        if (t >= P.T) break;
        const bf16* xr = p.x + static_cast<size_t>(t) * H;
        float acc = 0.0f;
        for (int h0 = lane; h0 < H; h0 += 128) {  // H % 128 == 0; loads issue ahead
            float v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = bf2f(xr[h0 + 32 * u]);
#pragma unroll
            for (int u = 0; u < 4; ++u) acc = fmaf(v[u], v[u], acc);  // v * v exact in fp32
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) acc = acc + __shfl_down_sync(0xffffffffu, acc, off);
        float rr = 0.0f;
        if (lane == 0)
            rr = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(acc, static_cast<float>(H)), p.eps)));
        rr = __shfl_sync(0xffffffffu, rr, 0);
        bf16* on = p.xn + static_cast<size_t>(t) * H;
#pragma unroll 4
        for (int h = lane; h < H; h += 32)
            on[h] = __float2bfloat16_rn(__fmul_rn(__fmul_rn(bf2f(xr[h]), rr), bf2f(p.gamma[h])));
    }
}

// The router weight chunk (and gamma) a CTA staged last stays in the ring for
// its next router task with the same chunk; any other use of the ring drops
// it.  The key (ctl->scratch[8..9]) is the chunk's global address, 0 = none.
constexpr int kWrKey = 8;
__device__ __forceinline__ void wr_cache_drop(Ctl* ctl) {
    if (wtid_() == 0) ctl->scratch[kWrKey] = ctl->scratch[kWrKey + 1] = 0;
}

// x_hat of a staged router tile in place, the arithmetic of norm_task (gamma
// staged too); warp w takes rows w, w + 8.  With `store` the rows also go to
// x_hat in global memory (for the permute and the shared expert).
__device__ __forceinline__ void norm_rows_staged(const MoeArgs& p, bf16* xs, const bf16* gs,
                                                 int t0, int nt, bool store) {
    const int H = p.H, warp = wtid_() >> 5, lane = wtid_() & 31;
    for (int t = warp; t < nt; t += kWorkers / 32) {
        bf16* xr = xs + static_cast<size_t>(t) * H;
        float acc = 0.0f;
        // H is a multiple of 128: blocks of 4 strided loads issue ahead of the
        // (ordered) accumulation
        for (int h0 = lane; h0 < H; h0 += 128) {
            float v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = bf2f(xr[h0 + 32 * u]);
#pragma unroll
            for (int u = 0; u < 4; ++u) acc = fmaf(v[u], v[u], acc);
        }
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) acc = acc + __shfl_down_sync(0xffffffffu, acc, off);
        float rr = 0.0f;
        if (lane == 0)
            rr = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(acc, static_cast<float>(H)), p.eps)));
        rr = __shfl_sync(0xffffffffu, rr, 0);
#pragma unroll 4
        for (int h = lane; h < H; h += 32)
            xr[h] = __float2bfloat16_rn(__fmul_rn(__fmul_rn(bf2f(xr[h]), rr), bf2f(gs[h])));
        if (store) {
            __syncwarp();
            uint4* dst = reinterpret_cast<uint4*>(p.xn + static_cast<size_t>(t0 + t) * H);
            const uint4* src = reinterpret_cast<const uint4*>(xr);
            for (int v = lane; v < H / 8; v += 32) dst[v] = src[v];
        }
    }
}

// Logits of router tile r for expert chunk c.  With staging, the token rows
// (one bulk copy) and the chunk's 8-expert weight blocks (TMA boxes) are
// copied into the ring, which the workers hold on lease for the task.  With
// several chunks the logits go to a global buffer and the chunk that brings
// the tile's counter to C does the top-k for the whole tile -- the same
// event-counter reduction as split-K.
__device__ __forceinline__ bool router_task(const MoeArgs& p, const MoePlan& P, int r, int c,
                                            uint8_t* smem, const Ring& ring, Ctl* ctl,
                                            const CUtensorMap* tm_wr, const WaitCtx& wc,
                                            uint32_t& sphase, uint32_t& seq) {
    const int E = p.E, H = p.H, k = p.k;
    float* lg = reinterpret_cast<float*>(smem);        // [16][E]
    int* hs = reinterpret_cast<int*>(smem + kHistOff);  // [E]
    int* sel_s = reinterpret_cast<int*>(smem + kSelOff);  // [nt * k]
    const int t0 = r * kRouterTile, nt = min(kRouterTile, P.T - t0);
    const int warp = wtid_() >> 5, lane = wtid_() & 31;
    const int e0 = c * P.EC, ec = P.EC;
    // fused block: a staged tile normalises its rows itself (NRN == 0);
    // otherwise it routes x_hat once every norm task is done
    const bool own_norm = p.gamma && P.NRN == 0;
    if (p.gamma && !own_norm) {
        if (wtid_() == 0) ctl->flag = ev_wait_geq(wc, &p.hdr->ev_norm, P.NRN, kWhereNorm) ? 1 : 0;
        worker_sync();
        if (!ctl->flag) return false;
        fence_proxy_async_global();  // x_hat rows written by generic stores, read by bulk copies
    }
    const bf16* xsrc = (p.gamma && !own_norm) ? p.xn : p.x;
    const bf16* xb = xsrc + static_cast<size_t>(t0) * H;
    const bf16* wb = p.wr + e0;
    int o = 0, rs = E, blk = 8;
    uint64_t tm = p.trace ? globaltimer_ns() : 0;
    if (P.stage) {
        const uint32_t xbytes = static_cast<uint32_t>(nt * H * 2);
        // the weight chunk sits after room for a full tile, at the same place for every tile
        const uint32_t xpad = (static_cast<uint32_t>(min(P.T, kRouterTile) * H * 2) + 1023u) & ~1023u;
        const int box = p.wr_box, hp = wr_rows_pad(H, box);
        const int eb0 = e0 >> 3, nb = ((e0 + ec + 7) >> 3) - eb0;
        uint8_t* wdst = ring.base + xpad;
        const uint32_t wbytes = P.wr_whole ? static_cast<uint32_t>(H) * static_cast<uint32_t>(E) * 2u
                                           : static_cast<uint32_t>(nb * hp * 16);
        uint8_t* gdst = wdst + wbytes;  // gamma (own norm)
        const uint32_t gbytes = own_norm ? static_cast<uint32_t>(H) * 2u : 0u;
        const uint64_t key = reinterpret_cast<uint64_t>(P.wr_whole ? p.wr : wb);
        const bool cached = static_cast<uint32_t>(ctl->scratch[kWrKey]) == static_cast<uint32_t>(key) &&
                            static_cast<uint32_t>(ctl->scratch[kWrKey + 1]) ==
                                static_cast<uint32_t>(key >> 32);
        worker_sync();  // every worker has read the key before it changes
        if (wtid_() == 0) {
            mbar_arrive_expect_tx(&ctl->sbar, xbytes + (cached ? 0u : wbytes + gbytes));
            bulk_g2s(ring.base, xb, xbytes, &ctl->sbar);
            if (!cached) {
                if (own_norm) bulk_g2s(gdst, p.gamma, gbytes, &ctl->sbar);
                if (P.wr_whole) {
                    bulk_g2s(wdst, p.wr, wbytes, &ctl->sbar);
                } else {
                    const uint64_t pol = policy_evict_last();
                    for (int b = 0; b < nb; ++b)
                        for (int h0 = 0; h0 < hp; h0 += box)
                            tma_load_2d(wdst + static_cast<size_t>(b * hp + h0) * 16, tm_wr,
                                        &ctl->sbar, (eb0 + b) * 8, h0, pol);
                }
                ctl->scratch[kWrKey] = static_cast<int>(static_cast<uint32_t>(key));
                ctl->scratch[kWrKey + 1] = static_cast<int>(static_cast<uint32_t>(key >> 32));
            }
        }
        if (!staging_wait(ctl, sphase, wc, seq)) return false;
        if (own_norm) {  // x -> x_hat in place; chunk 0 publishes the rows
            norm_rows_staged(p, reinterpret_cast<bf16*>(ring.base),
                             reinterpret_cast<const bf16*>(gdst), t0, nt, c == 0);
            worker_sync();
            if (c == 0) {
                fence_proxy_async_global();  // x_hat is read by TMA and bulk copies
                worker_sync();
                if (wtid_() == 0) {
                    __threadfence();
                    red_release_add(&p.hdr->ev_norm, 1);
                }
            }
        }
        tm = phase_mark(p, 0, tm);
        xb = reinterpret_cast<const bf16*>(ring.base);
        wb = reinterpret_cast<const bf16*>(wdst);
        if (P.wr_whole) {  // [H, E] as in global memory
            o = e0;
            rs = E;
            blk = 8;
        } else {
            o = e0 & 7;
            rs = 8;
            blk = hp * 8;
        }
    }
    float* out = P.C == 1 ? lg : p.logits + static_cast<size_t>(t0) * E;
    // A job is TB tokens x EBW experts on one warp.  The loop is latency-bound
    // rather than issue-bound, so few wide jobs beat one job per warp: EBW is
    // the widest block (<= 8) that divides the chunk (and E when the weight is
    // read in place, for aligned vector loads), TB is 4 tokens, or 1 when the
    // tile holds a single token.  Measured on GB300: 16 tokens x 2 experts as
    // four 4x2 jobs take 55 % of the time of eight 4x1 jobs; 1 token x 2
    // experts as one 1x2 job 60 % of the time of one 4x2 job.
    const int ew = (P.stage && !P.wr_whole) ? ec : (ec | E);
    const int ebw = ew % 8 == 0 ? 8 : (ew % 4 == 0 ? 4 : (ew % 2 == 0 ? 2 : 1));
    if (!P.stage) {
        router_logits_inplace(p.H, p.E, p.bias, xb, wb, o, rs, blk, nt, e0, ec, out);
    } else if (nt == 1) {
        if (ebw == 8)
            router_logits<8, 1>(p, xb, wb, o, rs, blk, nt, e0, ec, out);
        else if (ebw == 4)
            router_logits<4, 1>(p, xb, wb, o, rs, blk, nt, e0, ec, out);
        else if (ebw == 2)
            router_logits<2, 1>(p, xb, wb, o, rs, blk, nt, e0, ec, out);
        else
            router_logits<1, 1>(p, xb, wb, o, rs, blk, nt, e0, ec, out);
    } else {
        if (ebw == 8)
            router_logits<8, 4>(p, xb, wb, o, rs, blk, nt, e0, ec, out);
        else if (ebw == 4)
            router_logits<4, 4>(p, xb, wb, o, rs, blk, nt, e0, ec, out);
        else if (ebw == 2)
            router_logits<2, 4>(p, xb, wb, o, rs, blk, nt, e0, ec, out);
        else
            router_logits<1, 4>(p, xb, wb, o, rs, blk, nt, e0, ec, out);
    }
    worker_sync();
    tm = phase_mark(p, 1, tm);
    if (P.C > 1) {  // tile reduction through the tile's event counter
        if (wtid_() == 0) {
            __threadfence();
            ctl->flag = (atom_acq_rel_add(p.ev_tile + r, 1) == P.C - 1) ? 1 : 0;
        }
        worker_sync();
        if (!ctl->flag) return true;  // another chunk of this tile finishes it
        if (wtid_() == 0) p.ev_tile[r] = 0;  // every chunk arrived: reset for the next call
        for (int i = wtid_(); i < nt * E; i += kWorkers)
            lg[i] = __ldcg(p.logits + static_cast<size_t>(t0) * E + i);
        worker_sync();
        tm = phase_mark(p, 2, tm);
    }
    for (int e = wtid_(); e < E; e += kWorkers) hs[e] = 0;
    worker_sync();
    tm = phase_mark(p, 10, tm);
    // top-k per token (warp per token): order (logit desc, index asc).  A round
    // takes each lane's best remaining entry, then the warp's largest key and,
    // among lanes holding it, the smallest expert index (two redux
    // instructions).  The key is an order-preserving map of the fp32 logit,
    // with -0.0 taken as +0.0 (they tie).  After round j every lane holds the
    // j-th pick; lane j keeps it.  The rounds stay rolled: this code runs once
    // per call, often with cold instruction caches.
    for (int tt = warp; tt < nt; tt += kWorkers / 32) {
        const float* L = lg + tt * E;
        uint32_t key[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = lane + 32 * i;
            const float v = e < E ? L[e] : 0.0f;
            const uint32_t b = __float_as_uint(v == 0.0f ? 0.0f : v);
            key[i] = e < E ? ((b & 0x80000000u) ? ~b : (b | 0x80000000u)) : 0u;
        }
        uint32_t taken = 0;
        float myL = 0.0f;
        int myE = 0;
#pragma unroll 1
        for (int j = 0; j < k; ++j) {
            uint32_t bk = 0, bi = 0xffffffffu;  // this lane's best remaining (key, index)
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int e = lane + 32 * i;
                if (e < E && !((taken >> i) & 1u) && (bi == 0xffffffffu || key[i] > bk)) {
                    bk = key[i];
                    bi = static_cast<uint32_t>(e);
                }
            }
            const uint32_t kmax = __reduce_max_sync(0xffffffffu, bi == 0xffffffffu ? 0u : bk);
            const uint32_t win = __reduce_min_sync(0xffffffffu, (bi != 0xffffffffu && bk == kmax) ? bi : 0xffffffffu);
            if ((win & 31u) == static_cast<uint32_t>(lane)) taken |= 1u << (win >> 5);
            if (lane == j) {
                myE = static_cast<int>(win);
                myL = L[win];
            }
        }
        // gate weights over the k picks: exp(L_j - L_0) / sum_i exp(L_i - L_0)
        const float L0 = __shfl_sync(0xffffffffu, myL, 0);
        const float ex = lane < k ? expf(myL - L0) : 0.0f;
        float z = ex;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
        if (lane < k) {
            const int t = t0 + tt;
            p.idx[static_cast<size_t>(t) * k + lane] = myE;
            p.gw[static_cast<size_t>(t) * k + lane] = ex / z;
            sel_s[tt * k + lane] = myE;
            // one router tile: the expert's tokens as a mask (bit tt; its count is
            // the popcount, as a token picks an expert at most once); else counts
            if (P.R == 1)
                atomicOr(&hs[myE], 1 << tt);
            else
                atomicAdd(&hs[myE], 1);
        }
    }
    tm = phase_mark(p, 11, tm);
    worker_sync();
    tm = phase_mark(p, 3, tm);
    // the last router tile to finish runs the scan: no task waits for it.  A
    // single tile is its own last (its counts stay in smem for the scan).
    if (P.R > 1) {
        for (int e = wtid_(); e < E; e += kWorkers) p.hist[static_cast<size_t>(r) * E + e] = hs[e];
        worker_sync();
        if (wtid_() == 0) {
            __threadfence();
            ctl->flag = (atom_acq_rel_add(&p.hdr->ev_router, 1) == P.R - 1) ? 1 : 0;
        }
        worker_sync();
    }
    if (P.R == 1 && wtid_() == 0) ctl->flag = 1;
    worker_sync();
    tm = phase_mark(p, 4, tm);
    if (!ctl->flag) return true;
    return scan_task(p, P, smem, ring, ctl, wc, sphase, seq);  // hs, sel_s stay valid
}

// ------------------------------------------------------------------ SCAN

// Counts, offsets, expert row tiles, split choice, and the task queue, run by
// the last router tile to finish (every tile's histogram is visible through
// the acquire-release count).  The targets the later waits use (permute
// parts; F-tiles per chunk; the total number of output tiles) are all derived
// here, on the device, from the routing of this very call.  With one router
// tile the counts are this CTA's own histogram (smem) and the permutation
// indices follow from the top-k picks in smem (no row is copied: the gate/up
// tiles read the token rows in place); otherwise the per-tile histograms are
// staged in the ring and scanned per expert there.
__device__ __forceinline__ bool scan_task(const MoeArgs& p, const MoePlan& P, uint8_t* smem,
                                          const Ring& ring, Ctl* ctl, const WaitCtx& wc,
                                          uint32_t& sphase, uint32_t& seq) {
    const int E = p.E, k = p.k, R = P.R, T = P.T;
    uint64_t tm = p.trace ? globaltimer_ns() : 0;
    wr_cache_drop(ctl);  // the scan and the inline permute stage into the ring
    const int* hs1 = reinterpret_cast<const int*>(smem + kHistOff);  // R == 1: the counts
    int* cnt_s = reinterpret_cast<int*>(smem);  // [256]
    int* off_s = cnt_s + 256;                   // [257]
    int* n_s = off_s + 264;                     // [256]
    int* mtb_s = n_s + 256;                     // [257]
    uint32_t* tok_s = reinterpret_cast<uint32_t*>(mtb_s + 264);  // [256]: R == 1, tokens per expert
    const int RE = R * E;
    const bool staged = R > 1 && static_cast<size_t>(RE) * 4 <= ring.bytes;
    int* hs = reinterpret_cast<int*>(ring.base);
    if (R == 1) {  // the router tile's token masks
        for (int e = wtid_(); e < E; e += kWorkers) cnt_s[e] = __popc(hs1[e]);
    } else if (staged) {
        const int n4 = RE / 4;
        const int4* src = reinterpret_cast<const int4*>(p.hist);
        int4* dst = reinterpret_cast<int4*>(hs);
        constexpr int U = 8;
        for (int i = wtid_(); i < n4; i += kWorkers * U) {
            int4 v[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (i + u * kWorkers < n4) v[u] = __ldcg(src + i + u * kWorkers);
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (i + u * kWorkers < n4) dst[i + u * kWorkers] = v[u];
        }
        for (int i = n4 * 4 + wtid_(); i < RE; i += kWorkers) hs[i] = __ldcg(p.hist + i);
        worker_sync();
        for (int e = wtid_(); e < E; e += kWorkers) {
            int run = 0;
            for (int r = 0; r < R; ++r) {
                const int c = hs[r * E + e];
                hs[r * E + e] = run;
                run += c;
            }
            cnt_s[e] = run;
        }
    } else {
        for (int e = wtid_(); e < E; e += kWorkers) {
            int run = 0;
            for (int r = 0; r < R; ++r) {
                const int c = __ldcg(p.hist + static_cast<size_t>(r) * E + e);
                p.base[static_cast<size_t>(r) * E + e] = run;
                run += c;
            }
            cnt_s[e] = run;
        }
    }
    worker_sync();
    tm = phase_mark(p, 5, tm);
    const int FT = p.F / kTileM, HT = p.H / kTileM;
    // offsets and row-tile starts: one warp, a block of experts per lane and a
    // shuffle scan across lanes
    // Row tiles: an expert's rows split evenly over ceil(cnt / cap) tiles.  The
    // cap is kMoeNMax, or kMoeNSmall for experts whose weights are small
    // enough to be read again from L2 by each of their tiles: their tiles then
    // spread over more CTAs -- half of it up to 1024 routed rows, where a hot
    // expert's tiles are the last to finish (fine-grained shape, T = 128:
    // 162 -> 154 us; no change elsewhere).
    const bool small_e = 3ll * p.F * p.H * 2 <= kSmallExpertBytes;
    const int ncap = small_e ? (T * k <= 1024 ? kMoeNSmall / 2 : kMoeNSmall) : kMoeNMax;
    if (wtid_() < 32) {
        const int lane = wtid_(), per = ceil_div(E, 32);
        int csum = 0, msum = 0;
        for (int i = 0; i < per; ++i) {
            const int e = lane * per + i;
            if (e >= E) break;
            const int c = cnt_s[e];
            const int t = c == 0 ? 0 : ceil_div(c, ncap);  // the expert's row tiles
            const int n = c == 0 ? 0 : min(ncap, (ceil_div(c, t) + 15) / 16 * 16);
            n_s[e] = n;
            csum += c;
            msum += c == 0 ? 0 : ceil_div(c, n);
        }
        int cx = csum, mx = msum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int a = __shfl_up_sync(0xffffffffu, cx, off), b = __shfl_up_sync(0xffffffffu, mx, off);
            if (lane >= off) {
                cx += a;
                mx += b;
            }
        }
        cx -= csum;  // exclusive prefixes
        mx -= msum;
        for (int i = 0; i < per; ++i) {
            const int e = lane * per + i;
            if (e >= E) break;
            off_s[e] = cx;
            mtb_s[e] = mx;
            const int c = cnt_s[e];
            cx += c;
            mx += c == 0 ? 0 : ceil_div(c, n_s[e]);
        }
        if (lane == 31) {
            off_s[E] = cx;
            mtb_s[E] = mx;
        }
    }
    worker_sync();
    if (wtid_() == 0) {
        const int total_mt = mtb_s[E];
        // Wide down tiles (256 output columns: two weight boxes share one h
        // tile, so each expert's h rows are read half as often) when the row
        // tiles average 16 rows or more (measured on the Mixtral shape: 494
        // against 514 us at T = 128 and 479 against 494 us at T = 64, with
        // 128-column tiles the second figure).
        const int wide = (HT % 2 == 0 && T * k >= 16 * total_mt) ? 1 : 0;
        // split of the down projection: with few output tiles, the smallest
        // divisor of FT (<= 8) that gives the grid about four tasks a CTA (the
        // last wave of long tasks leaves CTAs idle); chunks keep >= 4 k-blocks,
        // and >= 8 once the grid has three tasks a CTA.  Wide tiles split in
        // two at most: measured on the Mixtral shape at T = 256, wide tiles in
        // 2 F-chunks take 494 us against 528 us for 128-column tiles in 4 and
        // 500 us for wide ones in 4 (their partials are twice the bytes).
        // A single token aims at two tasks a CTA (measured on the Mixtral
        // shape: 163 -> 157 us at T = 1; at T >= 2 the aim of four is faster).
        // Small tiles that already fill half the grid are not split: a split
        // adds a reduction chain (partials stored, counted, summed by the last
        // arriver, ~3 us) that a tile of <= 1 MB does not win back (measured
        // on the fine-grained shape: 85 -> 80 us at T = 1, 119 -> 111 us at
        // T = 8, without the splits of the down and gate/up tiles).
        const int G = p.num_ctas;
        int S = 1;
        const int down = total_mt * (wide ? HT / 2 : HT);
        const bool down_small = p.F * (wide ? 512 : 256) <= (1 << 20) && 2 * down >= G;
        if (T * k <= p.split_rows_cap && total_mt > 0 && down < 3 * G && !down_small) {
            int best = 1;
            for (int d = 2; d <= (wide ? 2 : kSplitMax); ++d) {
                if (!((p.split_mask >> d) & 1)) continue;
                const int kbc = p.F / kBlockK / d;
                if (down * best >= (T == 1 ? 2 : 3) * G && kbc < 8) break;
                best = d;
                if (down * d >= (T == 1 ? 2 : 4) * G) break;
            }
            S = best;
        }
        // K chunks of a gate/up tile: a small batch has few (weight-streaming)
        // tiles, so they are cut along K until the grid has two per CTA (three
        // measured 2 us slower on the Mixtral shape at T = 1)
        int KC = 1;
        const int gu = total_mt * FT;
        const bool gu_small = p.H * 512 <= (1 << 20) && 2 * gu >= G;
        while (!gu_small && KC < kGuSplitMax && gu * KC < 2 * G &&
               ((p.kc_mask >> (2 * KC)) & 1) && T * k * 2 * KC <= p.gu_cap)
            KC *= 2;
        ctl->scratch[0] = total_mt;
        ctl->scratch[1] = S;
        ctl->scratch[2] = KC;
        ctl->scratch[3] = wide;
    }
    worker_sync();
    tm = phase_mark(p, 6, tm);
    const int total_mt = ctl->scratch[0], S = ctl->scratch[1], KC = ctl->scratch[2];
    const int wide = ctl->scratch[3];
    // One router tile (R == 1): the gate/up tiles read the tile's token rows
    // straight from the layer's input -- no row is copied -- and keep, in the
    // epilogue, the columns of the tokens routed to their expert; the row
    // tile's entry carries those tokens (bit t, in the upper half of its N
    // word; an expert has one row tile, as T <= 16).
    const int* sel1 = reinterpret_cast<const int*>(smem + kSelOff);
    for (int e = wtid_(); e < E; e += kWorkers) {
        p.cnt[e] = cnt_s[e];
        p.off[e] = off_s[e];
        if (e == E - 1) p.off[E] = off_s[E];
        const int n = n_s[e];
        const uint32_t tok = R == 1 ? static_cast<uint32_t>(hs1[e]) : 0u;
        tok_s[e] = tok;
        p.e_tile[e] = make_int4(mtb_s[e], n, off_s[e], 0);
        for (int g = mtb_s[e], mt = 0; g < mtb_s[e + 1]; ++g, ++mt)
            p.g_info[g] = make_int4(e, off_s[e] + mt * n, min(n, cnt_s[e] - mt * n),
                                    static_cast<int>(static_cast<uint32_t>(n) | (tok << 16)));
    }
    if (R == 1) {
        for (int e = wtid_(); e < E; e += kWorkers) p.base[e] = off_s[e];
    } else if (staged) {
        for (int i = wtid_(); i < RE; i += kWorkers) p.base[i] = hs[i] + off_s[i % E];
    } else {
        for (int i = wtid_(); i < RE; i += kWorkers) p.base[i] += off_s[i % E];
    }
    tm = phase_mark(p, 7, tm);
    // The queue is implicit: every entry follows from the row tiles, S, KC and
    // the down-tile width, so the scan publishes those (and the row-tile table)
    // and each producer decodes the indices it claims (queue_task); nothing is
    // written per entry.  Order: [permute parts][gate/up tiles, by chunk]
    // [shared down tiles (fused block)][down tiles, by chunk][combine tasks].
    // A chunk c = (row tile g, F-chunk s) has u gate/up and d down tasks; every
    // down task comes after the gate/up tasks it waits for.  (Down tiles placed
    // right behind their chunk's gate/up tiles were measured slower on decode
    // and large batches: popped early, they stall their CTA on the dependency.)
    const int u = (FT / S) * KC, d = wide ? HT / 2 : HT, NCH = total_mt * S;
    const int total = P.NP + NCH * (u + d) + P.NSD + (P.NC > 1 ? P.NC : 0);
    worker_sync();  // the row-tile table and the permute bases are written
    if (wtid_() == 0) {
        p.hdr->total_mt = total_mt;
        p.hdr->split = S;
        p.hdr->gu_split = KC;
        p.hdr->q_wide = wide;
        p.hdr->q_total = total;
        __threadfence();
        st_release(&p.hdr->q_ready, 1);
    }
    if (R == 1) {  // after the publish: the permutation indices only (no row moves); the
                   // combine waits on their ev_perm release
        for (int i = wtid_(); i < T * k; i += kWorkers) {
            const int e = sel1[i], t = i / k;
            const int pp = off_s[e] + __popc(tok_s[e] & ((1u << t) - 1u));
            p.perm[pp] = i;
            p.pos[i] = pp;
            p.gpos[i] = mtb_s[e];
        }
        worker_sync();
        if (wtid_() == 0) {
            __threadfence();
            red_release_add(&p.hdr->ev_perm, 1);
        }
    }
    tm = phase_mark(p, 8, tm);
    return true;
}

// ------------------------------------------------------------------ PERMUTE

// Stable dispatch of router tile r: row (t, j) goes to off[e] + (rank of t
// among this call's tokens routed to e), and its x row is copied there.  The
// part's token rows come into the ring by bulk copy (the first batch is
// issued before the ranks are computed, so it flies meanwhile); each routed
// row then leaves with one bulk shared -> global copy.
__device__ __forceinline__ bool permute_rows(const MoeArgs& p, const MoePlan& P, int r, int i0,
                                             int i1, uint8_t* smem, const Ring& ring, Ctl* ctl,
                                             const WaitCtx& wc, uint32_t& sphase, uint32_t& seq) {
    const int k = p.k, E = p.E, H = p.H;
    const int t0 = r * kRouterTile, nt = min(kRouterTile, P.T - t0), nent = nt * k;
    int* ie = reinterpret_cast<int*>(smem + kPermOff);  // [128]
    int* slot = ie + 128;                               // [128]
    const int tl0 = i0 / k, ntok = i1 > i0 ? (i1 - 1) / k - tl0 + 1 : 0;
    const uint32_t rowb = static_cast<uint32_t>(H) * 2u;
    const int per = static_cast<int>(ring.bytes / rowb);  // rows a batch
    auto issue = [&](int c0) {  // worker thread 0: token rows tl0 + c0 .. of the part
        const int nc = min(per, ntok - c0);
        mbar_arrive_expect_tx(&ctl->sbar, nc * rowb);
        bulk_g2s(ring.base, (p.gamma ? p.xn : p.x) + static_cast<size_t>(t0 + tl0 + c0) * H,
                 nc * rowb, &ctl->sbar);
    };
    if ((p.gamma || p.ev_in) && wtid_() == 0) fence_proxy_async_global();  // generic stores
    if (ntok > 0 && wtid_() == 0) issue(0);
    for (int i = wtid_(); i < nent; i += kWorkers)
        ie[i] = __ldcg(p.idx + static_cast<size_t>(t0) * k + i);
    worker_sync();
    for (int i = i0 + wtid_(); i < i1; i += kWorkers) {
        const int e = ie[i], tl = i / k;
        int rank = 0;  // tokens before t in this tile routed to e (each at most once)
        for (int i2 = 0; i2 < tl * k; ++i2) rank += (ie[i2] == e);
        const int pp = __ldcg(p.base + static_cast<size_t>(r) * E + e) + rank;
        p.perm[pp] = t0 * k + i;
        p.pos[static_cast<size_t>(t0) * k + i] = pp;
        const int4 et = __ldcg(p.e_tile + e);  // the row's tile: first tile + offset / N
        p.gpos[static_cast<size_t>(t0) * k + i] = et.x + (pp - et.z) / et.y;
        slot[i] = pp;
    }
    for (int c0 = 0; c0 < ntok; c0 += per) {
        if (c0 > 0 && wtid_() == 0) issue(c0);
        if (!staging_wait(ctl, sphase, wc, seq)) return false;
        const int ia = max(i0, (tl0 + c0) * k), ib = min(i1, (tl0 + c0 + per) * k);
        for (int i = ia + wtid_(); i < ib; i += kWorkers)
            bulk_s2g(p.xp + static_cast<size_t>(slot[i]) * H,
                     ring.base + (i / k - tl0 - c0) * rowb, rowb);
        bulk_commit_wait_all();  // rows written (and the batch read) before the next one
        worker_sync();
    }
    if (ntok > 0) fence_proxy_async_global();  // the rows are read back by TMA
    worker_sync();
    return true;
}

// Permute task: part `part` of router tile r (entries split evenly in Q parts).
__device__ __forceinline__ bool permute_task(const MoeArgs& p, const MoePlan& P, int r, int part,
                                             uint8_t* smem, const Ring& ring, Ctl* ctl,
                                             const WaitCtx& wc, uint32_t& sphase, uint32_t& seq) {
    const int t0 = r * kRouterTile, nent = min(kRouterTile, P.T - t0) * p.k;
    wr_cache_drop(ctl);
    if (!permute_rows(p, P, r, part * nent / P.Q, (part + 1) * nent / P.Q, smem, ring, ctl, wc,
                      sphase, seq))
        return false;
    if (wtid_() == 0) {
        __threadfence();
        red_release_add(&p.hdr->ev_perm, 1);
    }
    return true;
}

// ------------------------------------------------------------------ COMBINE

// out[t] = bf16(sum_j w[t, j] * y[pos(t, j)]) in slot order -- in the fused
// block bf16(x[t] + sum_j w[t, j] * y[pos(t, j)] + ys[t]), summed in that order.
// The rows of a batch of tokens (k expert outputs, then x and ys in the
// block) are gathered into the ring with bulk copies, then summed from there.
__device__ __forceinline__ int combine_rows_per_token(const MoeArgs& p, const MoePlan& P) {
    return p.k + (p.gamma ? 1 : 0) + (P.MTS > 0 ? 1 : 0);
}

// A combine task's wait (bounded): only the row tiles that hold its tokens'
// k rows must be complete (every 128-column output tile of each), so
// combining overlaps the last down tiles of other row tiles.  Worker thread 0
// first acquires the permute (which wrote the rows' positions and tiles) and
// the shared expert; then each worker thread waits for one row's tile, all at
// once.  Returns the same decision to every worker.
__device__ __forceinline__ bool combine_wait_rows(const MoeArgs& p, const MoePlan& P, int t0,
                                                  int nt, Ctl* ctl, const WaitCtx& wc) {
    const int HT = p.H / kTileM, n = nt * p.k;
    if (wtid_() == 0)
        ctl->flag = (ev_wait_geq(wc, &p.hdr->ev_perm, P.NPW, kWherePerm) &&
                     (P.MTS == 0 || ev_wait_geq(wc, &p.hdr->ev_sdone, P.MTS * HT, kWhereY)))
                        ? 1 : 0;
    worker_sync();
    if (ctl->flag) {
        for (int i = wtid_(); i < n; i += kWorkers) {
            const int g = __ldcg(p.gpos + static_cast<size_t>(t0) * p.k + i);
            if (!ev_wait_geq(wc, p.ev_gdone + g, HT, kWhereY)) ctl->flag = 0;
        }
    }
    worker_sync();
    const bool ok = ctl->flag != 0;
    worker_sync();  // the flag is read before any later task writes it
    return ok;
}

__device__ __forceinline__ bool combine_task(const MoeArgs& p, const MoePlan& P, int c,
                                             uint8_t* smem, const Ring& ring, Ctl* ctl,
                                             const WaitCtx& wc, uint32_t& sphase, uint32_t& seq) {
    const int H = p.H, k = p.k;
    const int t0 = c * P.CT, nt = min(P.CT, P.T - t0), vpr = H / 8;
    wr_cache_drop(ctl);
    if (!combine_wait_rows(p, P, t0, nt, ctl, wc)) return false;
    fence_proxy_async_global();  // y rows written by other CTAs' generic stores
    const int rpt = combine_rows_per_token(p, P), hx = p.gamma ? 1 : 0, hs = P.MTS > 0 ? 1 : 0;
    const uint32_t rowb = static_cast<uint32_t>(H) * 2u;
    float* w_s = reinterpret_cast<float*>(smem);                   // [16 * k]
    int* pos_s = reinterpret_cast<int*>(smem) + kCombineTile * 8;  // [16 * k]
    for (int i = wtid_(); i < nt * k; i += kWorkers) {
        w_s[i] = __ldcg(p.gw + static_cast<size_t>(t0) * k + i);
        pos_s[i] = __ldcg(p.pos + static_cast<size_t>(t0) * k + i);
    }
    const int per = static_cast<int>(ring.bytes / (static_cast<uint32_t>(rpt) * rowb));
    if (wtid_() == 0 && nt > 0) mbar_arrive_expect_tx(&ctl->sbar, min(per, nt) * rpt * rowb);
    worker_sync();
    for (int b0 = 0; b0 < nt; b0 += per) {
        const int nb = min(per, nt - b0);
        for (int q = wtid_(); q < nb * rpt; q += kWorkers) {  // row q % rpt of token q / rpt
            const int tt = q / rpt, j = q % rpt, t = t0 + b0 + tt;
            const bf16* src = j < k ? p.y + static_cast<size_t>(pos_s[(b0 + tt) * k + j]) * H
                                    : (j == k && hx ? p.x : p.ys) + static_cast<size_t>(t) * H;
            bulk_g2s(ring.base + q * rowb, src, rowb, &ctl->sbar);
        }
        if (!staging_wait(ctl, sphase, wc, seq)) return false;
        for (int v = wtid_(); v < nb * vpr; v += kWorkers) {
            const int tt = v / vpr, cc = v % vpr;
            const uint8_t* rows = ring.base + tt * rpt * rowb;
            float acc[8];
            if (hx) {
                unpack8(reinterpret_cast<const uint4*>(rows + k * rowb)[cc], acc);  // residual
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
            }
            for (int j = 0; j < k; ++j) {  // fp32 sum in slot order j = 0 .. k-1
                const float wj = w_s[(b0 + tt) * k + j];
                float yv[8];
                unpack8(reinterpret_cast<const uint4*>(rows + j * rowb)[cc], yv);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj, yv[i], acc[i]);
            }
            if (hs) {  // the shared expert
                float yv[8];
                unpack8(reinterpret_cast<const uint4*>(rows + (k + hx) * rowb)[cc], yv);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = acc[i] + yv[i];
            }
            reinterpret_cast<uint4*>(p.out + static_cast<size_t>(t0 + b0 + tt) * H)[cc] = pack8(acc);
        }
        worker_sync();  // the batch is consumed before the ring is refilled
        if (wtid_() == 0 && b0 + per < nt)
            mbar_arrive_expect_tx(&ctl->sbar, min(per, nt - b0 - per) * rpt * rowb);
        worker_sync();
    }
    release_output(p, t0, nt);
    return true;
}

// All T (<= kCombineTile) tokens at once with plain loads: run by the last
// output tile to finish, inside its epilogue, while the ring may hold fills.
__device__ __forceinline__ void combine_inline(const MoeArgs& p, const MoePlan& P) {
    const int H = p.H, k = p.k, vpr = H / 8;
    for (int v = wtid_(); v < P.T * vpr; v += kWorkers) {
        const int t = v / vpr, cc = v % vpr;
        float acc[8];
        if (p.gamma) {
            unpack8(__ldcg(reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(t) * H) + cc), acc);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        }
        for (int j = 0; j < k; ++j) {  // fp32 sum in slot order j = 0 .. k-1
            const float wj = __ldcg(p.gw + static_cast<size_t>(t) * k + j);
            const int pp = __ldcg(p.pos + static_cast<size_t>(t) * k + j);
            float yv[8];
            unpack8(__ldcg(reinterpret_cast<const uint4*>(p.y + static_cast<size_t>(pp) * H) + cc), yv);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj, yv[i], acc[i]);
        }
        if (P.MTS > 0) {
            float yv[8];
            unpack8(__ldcg(reinterpret_cast<const uint4*>(p.ys + static_cast<size_t>(t) * H) + cc), yv);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = acc[i] + yv[i];
        }
        reinterpret_cast<uint4*>(p.out + static_cast<size_t>(t) * H)[cc] = pack8(acc);
    }
}

// ------------------------------------------------------------------ queue pop

// The producer's place in the task index space of the launch: layer l's
// tasks are [base, base + NS0 + q_total) -- its static prefix, then its queue
// (size known once its scan has run); the next layer's follow.
struct QCursor {
    int layer = 0, base = 0, qt = -1;
    int mt = 0, S = 1, KC = 1, wide = 0;  // the layer's published queue parameters
};

// Entry q of a layer's implicit queue (see scan_task for the order).
__device__ __forceinline__ TaskMsg queue_task(const MoeArgs& p, const MoePlan& P,
                                              const QCursor& cur, int q) {
    TaskMsg m{};
    if (q < P.NP) {  // permute part q % Q of router tile q / Q
        m.type = kTaskPermute;
        m.a = q / P.Q;
        m.b = q % P.Q;
        return m;
    }
    q -= P.NP;
    const int FT = p.F / kTileM, HT = p.H / kTileM, S = cur.S, KC = cur.KC;
    const int u = (FT / S) * KC, d = cur.wide ? HT / 2 : HT, NCH = cur.mt * S;
    const int flags = (S << 8) | (KC << 16) | (cur.wide << 24);
    if (q < NCH * u) {  // gate/up: row tile g, F-tile, K chunk
        const int c = q / u, r = q % u, g = c / S;
        m.type = kTaskGateUp | flags;
        m.a = g;
        m.b = (c % S) * (FT / S) + r / KC;
        m.c = r % KC;
        const int4 gi = __ldcg(p.g_info + g);
        m.e = gi.x, m.row0 = gi.y, m.rows = gi.z, m.n = gi.w & 0xffff;
        m.aux = static_cast<uint32_t>(gi.w) >> 16;
        return m;
    }
    q -= NCH * u;
    if (q < P.NSD) {  // fused block: shared down tile (row tile, F-chunk, output tile)
        const int mt = q / (P.SS * HT);
        m.type = kTaskShDown | (P.SS << 8);
        m.a = mt;
        m.b = (q % (P.SS * HT)) / HT;
        m.c = q % HT;
        m.row0 = mt * kWideNMax;
        m.rows = min(kWideNMax, P.T - m.row0);
        m.n = (m.rows + 15) / 16 * 16;
        return m;
    }
    q -= P.NSD;
    if (q < NCH * d) {  // down: row tile g, F-chunk, output tile (of 128, or 256 if wide)
        const int c = q / d, g = c / S;
        m.type = kTaskDown | flags;
        m.a = g;
        m.b = c % S;
        m.c = q % d;
        const int4 gi = __ldcg(p.g_info + g);
        m.e = gi.x, m.row0 = gi.y, m.rows = gi.z, m.n = gi.w & 0xffff;
        return m;
    }
    m.type = kTaskCombine;
    m.a = q - NCH * d;
    return m;
}

// Static-prefix task j of a layer: [norm][router][shared gate/up].
__device__ __forceinline__ TaskMsg static_task(const MoeArgs& p, const MoePlan& P, int j) {
    TaskMsg m{};
    if (j < P.NRN) {  // fused block: RMSNorm of router tile j's rows
        m.type = kTaskNorm;
        m.a = j;
        return m;
    }
    j -= P.NRN;
    const int nr = P.R * P.C;
    if (j < nr) {  // chunk-major: a CTA's next router task often reuses its staged chunk
        m.type = kTaskRouter;
        m.a = j % P.R;
        m.b = j / P.R;
        return m;
    }
    j -= nr;  // fused block: shared expert gate/up tiles (no routing needed)
    m.type = kTaskShGateUp;
    m.a = j / P.FTS;  // row tile
    m.b = j % P.FTS;  // F-tile
    m.row0 = m.a * kWideNMax;
    m.rows = min(kWideNMax, P.T - m.row0);
    m.n = (m.rows + 15) / 16 * 16;
    return m;
}

// While routing runs, HBM is idle.  A producer that has claimed gate/up
// queue entry q (after the permute parts) before the queue is published
// prefetches into L2 the first kSpecPrefetchKb of the gate/up weights the
// entry is predicted to need (plan.spec: expert q / (F/128), F-tile
// q % (F/128)), so the first wave of gate/up tiles reads them from L2.  A
// wrong prediction costs only bandwidth that was idle.
__device__ __forceinline__ void spec_prefetch(const MoeArgs& p, const MoeLayerMaps& M, int q) {
    const int FT = p.F / kTileM;
    if (q < 0 || q >= p.E * FT) return;
    const int row = (q / FT) * p.F + (q % FT) * kTileM;
    const int nkb = min(p.H / kBlockK, kSpecPrefetchKb / (2 * kABytes / 1024));
    for (int kb = 0; kb < nkb; ++kb) {
        tma_prefetch_l2(&M.wg, kb * kBlockK, row);
        tma_prefetch_l2(&M.wu, kb * kBlockK, row);
    }
}

// Producer thread: next task of this CTA (EXIT when every layer's tasks are
// taken or the launch aborted).  `claim` is a task index taken ahead of time
// (or -1); claims only grow, so the cursor only moves forward.  With `nowait`
// a claim that falls in a queue not yet published gives kTaskNone (the claim
// stays the caller's) instead of waiting for the scan.
template <bool kChain>
__device__ __forceinline__ TaskMsg pop_task(const MoeLaunchOf<kChain>& Lc, const MoePlan* plans,
                                            const WaitCtx& wc, int claim, QCursor& cur,
                                            bool nowait = false) {
    TaskMsg m{};
    m.type = kTaskExit;
    if (aborted(wc) || plans[0].R == 0) return m;  // T == 0: no task at all
    const int i = claim >= 0 ? claim : atomicAdd(&Lc.a[0].hdr->q_head, 1);
    for (;;) {
        const int l = kChain ? cur.layer : 0;
        const MoeArgs& p = Lc.a[l];
        const MoePlan& P = plans[l];
        const int j = i - cur.base;
        if (j < P.NS0) {
            m = static_task(p, P, j);
            break;
        }
        if (cur.qt < 0) {
            if (nowait && ld_acquire(&p.hdr->q_ready) < 1) {
                m.type = kTaskNone;
                return m;
            }
            if (P.spec && ld_acquire(&p.hdr->q_ready) < 1)
                spec_prefetch(p, Lc.m[kChain ? cur.layer : 0], j - P.NS0 - P.NP);
            if (!ev_wait_geq(wc, &p.hdr->q_ready, 1, kWhereQueue)) return m;
            cur.qt = ld_relaxed(&p.hdr->q_total);
            cur.mt = ld_relaxed(&p.hdr->total_mt);
            cur.S = ld_relaxed(&p.hdr->split);
            cur.KC = ld_relaxed(&p.hdr->gu_split);
            cur.wide = ld_relaxed(&p.hdr->q_wide);
        }
        if (j < P.NS0 + cur.qt) {
            m = queue_task(p, P, cur, j - P.NS0);
            break;
        }
        if (!kChain || cur.layer + 1 >= Lc.nl) return m;  // every layer's tasks are taken
        cur.base += P.NS0 + cur.qt;
        ++cur.layer;
        cur.qt = -1;
    }
    if (kChain) m.type |= cur.layer << kLayerShift;
    return m;
}

// ------------------------------------------------------------------ the kernel

// kChain: more than one layer.  A single layer takes every argument from
// layer 0 at fixed parameter offsets; a chain indexes the layer per task.
template <bool kChain>
__global__ void __launch_bounds__(kThreads, 1) moe_megakernel(
    const __grid_constant__ MoeLaunchOf<kChain> Lc) {
    extern __shared__ uint8_t smem_raw[];
    const uint64_t t_start = globaltimer_ns();
    Ring ring;
    uint8_t* scratch;
    Ctl* ctl = cta_setup(smem_raw, kMoeScratch, ring, &scratch);
    const MoeArgs& p0 = Lc.a[0];  // the launch's header: queue head, status, abort, exit count
    const WaitCtx wc{p0.hdr, p0.timeout_ns};
    const uint32_t tmem = ctl->tmem_base;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) trace_rec(p0, 0, 2, 0, 0, t_start, globaltimer_ns());

#ifdef ET_FIXED_T
    // A build specialised for one token count (the per-batch-size builds the
    // warm-up comparison times): T is a compile-time constant, the host and
    // device counts are ignored.
    int T = ET_FIXED_T;
#else
    int T = p0.T_host;
    if (p0.d_T) T = *reinterpret_cast<const volatile int32_t*>(p0.d_T);
#endif
    if (T < 0 || T > p0.T_max) {
        if (blockIdx.x == 0 && threadIdx.x == 0) raise_error(wc, ET_ERR_BOUNDS, kWhereBoundsT);
        T = 0;
    }
    // every layer's plan, once per CTA (shared memory, read by every role)
    MoePlan* plans = reinterpret_cast<MoePlan*>(scratch + kPlanOff);
    if (threadIdx.x == 0) ctl->scratch[kWrKey] = ctl->scratch[kWrKey + 1] = 0;
    if (static_cast<int>(threadIdx.x) < Lc.nl)
        plans[threadIdx.x] =
            moe_plan(Lc.a[threadIdx.x], T, static_cast<int>(gridDim.x), ring.bytes);
    __syncthreads();
    const int FT = p0.F / kTileM, HT = p0.H / kTileM;  // shapes shared by every layer

    auto is_gemm = [](int type) {
        return type == kTaskGateUp || type == kTaskDown || type == kTaskShGateUp ||
               type == kTaskShDown;
    };
    auto gemm_of = [&](const TaskMsg& m) {
        const int type = m.type & 0xff, S = (m.type >> 8) & 0xff, KC = (m.type >> 16) & 0xff;
        const int l = kChain ? layer_of(m) : 0;
        const MoeArgs& p = Lc.a[l];
        const MoeLayerMaps& M = Lc.m[l];
        const MoePlan& P = plans[l];
        if (type == kTaskShGateUp)  // shared expert over the rows of x_hat
            return GemmTask{&M.sg, &M.su, &M.xn, nullptr, m.b * kTileM, m.row0, 0,
                            p.H / kBlockK, m.n, &p.hdr->ev_norm, P.R, kWhereNorm};
        if (type == kTaskShDown) {
            const int fch = p.Fs / S;
            return GemmTask{&M.sd, nullptr, &M.hs, nullptr, m.c * kTileM, m.row0,
                            m.b * (fch / kBlockK), fch / kBlockK, m.n,
                            &p.ev_hs[m.a * kSplitMax + m.b], P.FTS / S, kWhereH};
        }
        if (type == kTaskGateUp) {
            const int nkb = p.H / kBlockK / KC;
            if (P.R == 1) {  // the router tile's rows (x_hat in a block), all 16 columns
                const int* dep = p.gamma ? &p.hdr->ev_norm : p.ev_in;
                return GemmTask{&M.wg, &M.wu, &M.xr, nullptr, m.e * p.F + m.b * kTileM, 0,
                                m.c * nkb, nkb, kRouterTile, dep, p.gamma ? 1 : P.T,
                                p.gamma ? kWhereNorm : kWhereInput};
            }
            return GemmTask{&M.wg, &M.wu, &M.xp, p.b_wide ? &M.xp64 : nullptr,
                            m.e * p.F + m.b * kTileM, m.row0, m.c * nkb, nkb, m.n,
                            &p.hdr->ev_perm, P.NPW, kWherePerm};
        }
        const int fchunk = p.F / S, wide = (m.type >> 24) & 1;
        return GemmTask{&M.wd, wide ? &M.wd : nullptr, &M.h, p.b_wide ? &M.h64 : nullptr,
                        m.e * p.H + m.c * (kTileM << wide), m.row0, m.b * (fchunk / kBlockK),
                        fchunk / kBlockK, m.n, &p.ev_h[m.a * kSplitMax + m.b], FT / S, kWhereH,
                        wide ? kTileM : 0};
    };

    if (warp == 0) {
        if (lane == 0) {  // producer: pop, hand over, load (one GEMM task of lookahead)
            const uint64_t pol_w = policy_evict_first(), pol_b = policy_evict_last();
            ProdState ps;
            QCursor cur;
            int claim = -1, sent = 0;
            Flight fc, fn;                     // the current task; the one looked ahead
            bool has_next = false, end = false;  // end: EXIT handed during a lookahead
            // hand a task to the MMA issuer and the workers (the slot is free)
            auto hand = [&](const TaskMsg& m) {
                const int slot = sent % kTaskRing;
                ctl->tq[slot] = m;
                mbar_arrive(&ctl->tq_full[slot]);
                ++sent;
            };
            auto slot_free = [&]() {
                return mbar_try_wait(&ctl->tq_empty[sent % kTaskRing],
                                     ((sent / kTaskRing) & 1) ^ 1);
            };
            // while the current task waits on its dependency: take the next
            // task if it can be decoded and handed over without waiting, and
            // post the weights of a GEMM task into free ring space.  A SIMT task
            // (it leases the whole ring) or EXIT ends the lookahead.
            auto idle = [&]() {
                if (!has_next) {
                    if (end || *reinterpret_cast<volatile int32_t*>(&ctl->ring_ret) <
                                   static_cast<int32_t>(ps.leases))
                        return;
                    if (!slot_free()) return;
                    const uint64_t tp = globaltimer_ns();
                    const TaskMsg m = pop_task<kChain>(Lc, plans, wc, claim, cur, true);
                    const int type = m.type & 0xff;
                    if (type == kTaskNone) return;
                    claim = -1;
                    hand(m);
                    if (type == kTaskExit) {
                        end = true;
                        return;
                    }
                    if (!is_gemm(type)) {
                        ++ps.leases;
                        trace_rec(p0, type, 0, m.a, m.b, tp, globaltimer_ns());
                        return;
                    }
                    claim = atomicAdd(&p0.hdr->q_head, 1);
                    flight_begin(fn, gemm_of(m), type, m.a, m.b, tp);
                    has_next = true;
                }
                flight_post_nowait(fn, ring, ctl, ps, pol_w, pol_b);
            };
            for (;;) {
                if (has_next) {
                    fc = fn;
                    has_next = false;
                } else {
                    if (end) break;
                    // a SIMT task still out on lease: take no further task before it
                    // is done, so SIMT work spreads over the CTAs that are free
                    if (!ring_lease_wait(ctl, ps, wc)) break;
                    const uint64_t tp = globaltimer_ns();
                    const TaskMsg m = pop_task<kChain>(Lc, plans, wc, claim, cur);
                    claim = -1;
                    if (!mbar_wait(wc, &ctl->tq_empty[sent % kTaskRing],
                                   ((sent / kTaskRing) & 1) ^ 1, kWhereQueue))
                        break;
                    hand(m);
                    const int type = m.type & 0xff;
                    if (type == kTaskExit) break;
                    if (!is_gemm(type)) {
                        ++ps.leases;  // a SIMT task holds the ring until the workers return it
                        trace_rec(p0, type, 0, m.a, m.b, tp, globaltimer_ns());
                        continue;
                    }
                    // claim the next task now: the atomic's latency hides behind the loads
                    claim = atomicAdd(&p0.hdr->q_head, 1);
                    flight_begin(fc, gemm_of(m), type, m.a, m.b, tp);
                    flight_post_nowait(fc, ring, ctl, ps, pol_w, pol_b);
                }
                if (!flight_wait(fc, ring, ctl, ps, wc, pol_w, pol_b, idle)) break;
                if (!flight_finish(fc, ring, ctl, ps, wc, pol_w, pol_b)) break;
                trace_rec(p0, fc.type, 0, fc.a, fc.b, fc.t_pop, globaltimer_ns());
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {  // MMA issuer
            MmaState ms;
            for (int i = 0;; ++i) {
                const int slot = i % kTaskRing;
                if (!mbar_wait(wc, &ctl->tq_full[slot], (i / kTaskRing) & 1, kWhereQueue)) break;
                const TaskMsg m = ctl->tq[slot];
                mbar_arrive(&ctl->tq_empty[slot]);
                const int type = m.type & 0xff;
                if (type == kTaskExit) break;
                if (!is_gemm(type)) continue;
                if (p0.trace) {  // role 5: one record per fill, posted .. landed
                    auto ftr = [&](int u, uint64_t tp, uint64_t tl) {
                        trace_rec(p0, type, 5, m.a, u, tp, tl);
                    };
                    if (!mma_task(gemm_of(m), ring, ctl, ms, tmem, wc, ftr)) break;
                } else if (!mma_task(gemm_of(m), ring, ctl, ms, tmem, wc)) {
                    break;
                }
            }
        }
        __syncwarp();
    } else if (warp >= kEpiWarp0) {  // workers: epilogues and SIMT tasks
        const int q = warp & 3, half = (warp - kEpiWarp0) >> 2, wtid = wtid_();  // TMEM quadrant, column half
        const int H = p0.H, F = p0.F;
        EpiState es;
        uint32_t sphase = 0;
        for (int i = 0;; ++i) {
            const int slot = i % kTaskRing;
            if (!worker_wait(ctl, &ctl->tq_full[slot], (i / kTaskRing) & 1, wc, kWhereQueue, es.seq))
                break;
            const TaskMsg m = ctl->tq[slot];
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->tq_empty[slot]);
            const int type = m.type & 0xff, S = (m.type >> 8) & 0xff, KC = (m.type >> 16) & 0xff;
            const int wide = (m.type >> 24) & 1;
            if (type == kTaskExit) break;
            const int l = kChain ? layer_of(m) : 0;
            const MoeArgs& p = Lc.a[l];
            const MoePlan& P = plans[l];
            TraceScope trace_scope{p, type, m.a, m.b, p.trace ? globaltimer_ns() : 0ull,
                                   p.trace != nullptr && wtid == 0};
            if (!is_gemm(type)) {  // SIMT task on the leased ring
                bool ok = true;
                if (type == kTaskNorm) {
                    ok = wait_input(p, P, m.a, ctl, wc);
                    if (ok) {
                        norm_task(p, P, m.a);
                        fence_proxy_async_global();  // x_hat is read by TMA and bulk copies
                        worker_sync();
                        if (wtid == 0) {
                            __threadfence();
                            red_release_add(&p.hdr->ev_norm, 1);
                        }
                    }
                } else if (type == kTaskRouter)
                    ok = ((p.gamma && P.NRN > 0) || wait_input(p, P, m.a, ctl, wc)) &&
                         router_task(p, P, m.a, m.b, scratch, ring, ctl, &Lc.m[l].wr, wc, sphase,
                                     es.seq);
                else if (type == kTaskPermute)
                    ok = permute_task(p, P, m.a, m.b, scratch, ring, ctl, wc, sphase, es.seq);
                else
                    ok = combine_task(p, P, m.a, scratch, ring, ctl, wc, sphase, es.seq);
                if (!ok) break;
                ring_return(ctl);
                continue;
            }
            const bool two = type == kTaskGateUp || type == kTaskShGateUp || wide;
            wr_cache_drop(ctl);  // the tile's fills went through the ring
            uint32_t acc, acc1;
            if (!epi_acquire(ctl, es, two, m.n, tmem, wc, acc, acc1)) break;
            if (p.trace && wtid == 0)
                trace_rec(p, type, 6, m.a, m.b, trace_scope.t0, globaltimer_ns());
            const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
            const uint32_t lane_base = acc + lane_off;
            const int row0 = m.row0, rows = m.rows, n = m.n;
            if (type == kTaskShGateUp) {  // shared expert: hs = bf16(silu(g) * u)
                const int Fs = p.Fs, ft = m.b, f = ft * kTileM + q * 32 + lane;
                for (int c0 = half * 16; c0 < n; c0 += 32) {
                    float gv[16], uv[16];
                    tmem_ld16(lane_base + c0, gv);
                    tmem_ld16(acc1 + lane_off + c0, uv);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        if (c0 + c < rows)
                            p.hs[static_cast<size_t>(row0 + c0 + c) * Fs + f] =
                                __float2bfloat16_rn(silu_mul(gv[c], uv[c]));
                }
                epi_release(ctl, es, true, n);
                fence_proxy_async_global();  // hs is read back by TMA
                worker_sync();
                if (wtid == 0) {
                    __threadfence();
                    red_release_add(&p.ev_hs[m.a * kSplitMax + ft / (P.FTS / P.SS)], 1);
                }
                continue;
            }
            if (type == kTaskShDown) {  // shared expert: ys (or an fp32 partial of F-chunk s)
                const int s = m.b, ht = m.c, hh = ht * kTileM + q * 32 + lane;
                const int cap = p.split_rows_cap;
                for (int c0 = half * 16; c0 < n; c0 += 32) {
                    float v[16];
                    tmem_ld16(lane_base + c0, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        if (c0 + c >= rows) continue;
                        const size_t row = static_cast<size_t>(row0 + c0 + c);
                        if (S == 1)
                            p.ys[row * H + hh] = __float2bfloat16_rn(v[c]);
                        else
                            p.partial_s[(static_cast<size_t>(s) * cap + row) * H + hh] = v[c];
                    }
                }
                epi_release(ctl, es, false, n);
                fence_proxy_async_global();  // ys is gathered by bulk copies in the combine
                worker_sync();
                bool done = true;
                if (S > 1) {
                    int* ev = p.ev_ys + m.a * HT + ht;
                    if (wtid == 0) {
                        __threadfence();
                        ctl->flag = (atom_acq_rel_add(ev, 1) == S - 1) ? 1 : 0;
                    }
                    worker_sync();
                    done = ctl->flag != 0;
                    if (done) {  // last arriver: sum the partials in chunk order
                        if (wtid == 0) *ev = 0;  // every chunk arrived: reset for the next call
                        reduce_slice4(p.partial_s, static_cast<size_t>(cap) * H, H, S, row0,
                                      row0 + rows, ht * kTileM, p.ys, H);
                        fence_proxy_async_global();
                        worker_sync();
                    }
                }
                if (done && wtid == 0) {
                    __threadfence();
                    red_release_add(&p.hdr->ev_sdone, 1);
                }
                continue;
            }
            if (type == kTaskGateUp) {
                const int ft = m.b;
                const int f = ft * kTileM + q * 32 + lane;
                // K-split tile: fp32 partials of chunk m.c, rows of this call
                const size_t tk = static_cast<size_t>(P.T) * p.k;
                float* gpart = p.gu_part + (static_cast<size_t>(m.c) * tk) * F;
                float* upart = gpart + static_cast<size_t>(p.gu_cap) * F;
                // one router tile: column c is token c; a token routed to this
                // expert goes to its permuted row (its rank among them)
                const uint32_t tok = m.aux;
                for (int c0 = half * 16; c0 < n; c0 += 32) {
                    float gv[16], uv[16];
                    tmem_ld16(lane_base + c0, gv);
                    tmem_ld16(acc1 + lane_off + c0, uv);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        int rr = c0 + c;
                        if (tok) {
                            if (!((tok >> rr) & 1u)) continue;
                            rr = __popc(tok & ((1u << rr) - 1u));
                        } else if (rr >= rows) {
                            continue;
                        }
                        const size_t r = static_cast<size_t>(row0 + rr);
                        if (KC == 1) {
                            p.h[r * F + f] = __float2bfloat16_rn(silu_mul(gv[c], uv[c]));
                        } else {
                            gpart[r * F + f] = gv[c];
                            upart[r * F + f] = uv[c];
                        }
                    }
                }
                epi_release(ctl, es, true, n);
                if (KC > 1) {  // the chunk that completes the tile sums the partials
                    int* ev = p.ev_gu + m.a * FT + ft;
                    worker_sync();
                    if (wtid == 0) {
                        __threadfence();
                        ctl->flag = (atom_acq_rel_add(ev, 1) == KC - 1) ? 1 : 0;
                    }
                    worker_sync();
                    if (!ctl->flag) continue;
                    if (wtid == 0) *ev = 0;  // every chunk arrived: reset for the next call
                    const float* g0 = p.gu_part;
                    const float* u0 = p.gu_part + static_cast<size_t>(p.gu_cap) * F;
                    for (int j = wtid; j < rows * kTileM; j += kWorkers) {
                        const size_t r = static_cast<size_t>(row0 + j / kTileM);
                        const int ff = ft * kTileM + j % kTileM;
                        float gs = 0.0f, us = 0.0f;  // chunk order kc = 0 .. KC-1
                        for (int kc = 0; kc < KC; ++kc) {
                            const size_t o = (static_cast<size_t>(kc) * tk + r) * F + ff;
                            gs += __ldcg(g0 + o);
                            us += __ldcg(u0 + o);
                        }
                        p.h[r * F + ff] = __float2bfloat16_rn(silu_mul(gs, us));
                    }
                }
                fence_proxy_async_global();  // h is read back by TMA
                worker_sync();
                if (wtid == 0) {
                    const bool skip = p.fault_mode == 1 && m.a * FT + ft == p.fault_arg;
                    __threadfence();
                    if (!skip) red_release_add(&p.ev_h[m.a * kSplitMax + ft / (FT / S)], 1);
                }
                continue;
            }
            // DOWN: y (S == 1) or an fp32 partial of F-chunk s (partials [row][S]);
            // a wide tile holds output columns [256 ht, +128) in acc and
            // [256 ht + 128, +128) in acc1
            const int s = m.b, ht = m.c;
            for (int w = 0; w <= wide; ++w) {
                const int hh = ht * (kTileM << wide) + w * kTileM + q * 32 + lane;
                const uint32_t ab = (w ? acc1 : acc) + lane_off;
                for (int c0 = half * 16; c0 < n; c0 += 32) {
                    float v[16];
                    tmem_ld16(ab + c0, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        if (c0 + c >= rows) continue;
                        const size_t row = static_cast<size_t>(row0 + c0 + c);
                        if (S == 1)
                            p.y[row * H + hh] = __float2bfloat16_rn(v[c]);
                        else
                            p.partial[(row * S + s) * H + hh] = v[c];
                    }
                }
            }
            epi_release(ctl, es, two, n);
            fence_proxy_async_global();  // y is gathered by bulk copies in the combine
            worker_sync();  // the tile's stores are done
            bool done = true;
            if (S > 1) {
                if (wtid == 0) {
                    __threadfence();
                    ctl->flag = (atom_acq_rel_add(&p.ev_y[m.a * HT + ht], 1) == S - 1) ? 1 : 0;
                }
                worker_sync();
                done = ctl->flag != 0;
                if (done) {  // last arriver: sum the partials in chunk order
                    for (int w = 0; w <= wide; ++w)
                        reduce_slice4(p.partial, static_cast<size_t>(H), S * H, S, row0,
                                      row0 + rows, ht * (kTileM << wide) + w * kTileM, p.y, H);
                    fence_proxy_async_global();
                    worker_sync();
                }
            }
            const int ntiles = 1 + wide;  // 128-column output tiles completed
            if (done && P.NC > 1) {  // the combine tasks wait on the row tile's counter
                if (wtid == 0) {
                    __threadfence();
                    red_release_add(p.ev_gdone + m.a, ntiles);
                }
            } else if (done) {  // one combine: the last output tile to finish runs it
                if (wtid == 0) {
                    __threadfence();
                    const int target = ld_relaxed(&p.hdr->total_mt) * HT;
                    bool last = atom_acq_rel_add(&p.hdr->ev_ydone, ntiles) == target - ntiles;
                    // it also needs the permutation indices (a single router tile writes
                    // them after its gate/up tiles may have started) and the shared
                    // expert's output tiles
                    if (last)
                        last = ev_wait_geq(wc, &p.hdr->ev_perm, P.NPW, kWherePerm) &&
                               (P.MTS == 0 || ev_wait_geq(wc, &p.hdr->ev_sdone, P.MTS * HT, kWhereY));
                    ctl->flag = last ? 1 : 0;
                }
                worker_sync();
                const bool go = ctl->flag != 0;
                worker_sync();  // the flag is read before any later task writes it
                if (go) {
                    combine_inline(p, P);
                    release_output(p, 0, P.T);
                }
            }
        }
    }

    const uint64_t t_exit = globaltimer_ns();
    const bool aborted_run = ld_relaxed(&p0.hdr->abort) != 0;
    cta_teardown(ctl, aborted_run);
    if (threadIdx.x == 0) trace_rec(p0, 0, 3, 0, 0, t_exit, globaltimer_ns());

    // Exit protocol: the last CTA out returns every counter to zero.
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        ctl->flag = (atomicAdd(&p0.hdr->exit_count, 1) == static_cast<int>(gridDim.x) - 1) ? 1 : 0;
    }
    __syncthreads();
    if (ctl->flag) {
        __threadfence();
        const bool aborted_all = ld_relaxed(&p0.hdr->abort) != 0;
        for (int l = 0; l < (kChain ? Lc.nl : 1); ++l) {
            const MoeArgs& p = Lc.a[l];
            const MoePlan& P = plans[l];
            const bool clean = !aborted_all && ld_relaxed(&p.hdr->q_ready) != 0;
            const int mt = clean ? ld_relaxed(&p.hdr->total_mt) : p.mt_max;
            for (int i = threadIdx.x; i < mt * kSplitMax; i += kThreads) p.ev_h[i] = 0;
            for (int i = threadIdx.x; i < mt * HT; i += kThreads) p.ev_y[i] = 0;
            for (int i = threadIdx.x; i < mt; i += kThreads) p.ev_gdone[i] = 0;
            const int mts = clean ? P.MTS : p.mts_max;
            for (int i = threadIdx.x; i < mts * kSplitMax; i += kThreads) p.ev_hs[i] = 0;
            if (p.ev_tok) {
                const int nr = clean ? P.R : p.r_max;
                for (int i = threadIdx.x; i < nr; i += kThreads) p.ev_tok[i] = 0;
            }
            if (!clean) {  // self-resetting counters an aborted launch may have left behind
                for (int i = threadIdx.x; i < p.mt_max * FT; i += kThreads) p.ev_gu[i] = 0;
                for (int i = threadIdx.x; i < p.r_max; i += kThreads) p.ev_tile[i] = 0;
                for (int i = threadIdx.x; i < p.mts_max * HT; i += kThreads) p.ev_ys[i] = 0;
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int l = 0; l < (kChain ? Lc.nl : 1); ++l) {
                EtHeader* hd = Lc.a[l].hdr;
                hd->q_head = 0;
                hd->q_ready = 0;
                hd->q_total = 0;
                hd->total_mt = 0;
                hd->ev_router = 0;
                hd->ev_perm = 0;
                hd->ev_ydone = 0;
                hd->split = 0;
                hd->gu_split = 0;
                hd->q_wide = 0;
                hd->ev_norm = 0;
                hd->ev_sdone = 0;
                hd->abort = 0;
            }
            __threadfence();
            p0.hdr->exit_count = 0;
        }
    }
}

int moe_smem_bytes() { return smem_bytes_for(kMoeScratch); }
int moe_ring_bytes() { return ring_bytes_for(kMoeScratch); }

// Host-side launch (called by the C ABI after validation).
cudaError_t launch_moe(const MoeArgs* a, const CUtensorMap* maps, int nl, int grid, int smem,
                       cudaStream_t stream) {
    static_assert(sizeof(MoeLayerMaps) == kMapsPerLayer * sizeof(CUtensorMap), "maps of a layer");
    if (nl < 1 || nl > kMaxLayers) return cudaErrorInvalidValue;
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
    if (nl == 1) {
        MoeLaunchOf<false> L;
        memset(&L, 0, sizeof(L));
        memcpy(&L.m[0], maps, sizeof(MoeLayerMaps));
        L.a[0] = a[0];
        L.nl = 1;
        return cudaLaunchKernelEx(&cfg, moe_megakernel<false>, L);
    }
    MoeLaunchOf<true> L;
    memset(&L, 0, sizeof(L));
    for (int l = 0; l < nl; ++l) {
        memcpy(&L.m[l], maps + kMapsPerLayer * l, sizeof(MoeLayerMaps));
        L.a[l] = a[l];
    }
    L.nl = nl;
    return cudaLaunchKernelEx(&cfg, moe_megakernel<true>, L);
}

cudaError_t prepare_moe(int smem) {
    cudaError_t e = cudaFuncSetAttribute(moe_megakernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(moe_megakernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem);
}

}  // namespace et
