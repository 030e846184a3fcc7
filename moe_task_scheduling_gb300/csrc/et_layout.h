// et_layout.h -- workspace header, kernel argument blocks and tiling
// constants shared by the host launcher and the kernels of libetmoe.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/etmoe.h"

namespace et {

using bf16 = __nv_bfloat16;

// ---------------------------------------------------------------- tiling constants

constexpr int kThreads = 320;        // 10 warps: 0 TMA, 1 MMA/TMEM, 2-9 workers
constexpr int kEpiWarp0 = 2;         // worker warp w reads TMEM lanes 32*(w%4) ..
constexpr int kTileM = 128;          // weight rows per tile (UMMA M)
constexpr int kBlockK = 64;          // bf16 elements per k-block = one 128-byte swizzle row
constexpr int kABytes = kTileM * kBlockK * 2;   // 16 KB weight tile
constexpr int kBBoxRows = 16;        // activation rows per TMA box
constexpr int kBBoxRowsWide = 64;    // activation rows per wide TMA box
constexpr int kTmemCols = 512;       // accumulator 0 at column 0, accumulator 1 at 256
constexpr int kAcc1Col = 256;
constexpr int kSmemLimit = 232448;   // 227 KB of opt-in dynamic shared memory per CTA
constexpr int kSplitMax = 8;         // largest split of the MoE / MLP down projection

// MoE
constexpr int kMoeNMax = 256;        // token rows per expert tile (UMMA N)
// Row-tile cap of an expert whose weights (gate, up, down) are at most
// kSmallExpertBytes: its tiles re-read them from L2, and more, shorter tiles
// balance the grid (measured on the fine-grained shape, 9.4 MB an expert:
// T = 256 / 512 / 1024 / 4096 from 191 / 228 / 310 / 725 us with 256-row
// tiles to 174 / 213 / 300 / 718 us; a cap of 64 lost at T >= 256; the
// Mixtral-shaped experts, 352 MB each, keep 256-row tiles: 128-row tiles
// re-read them from HBM, 538 -> 715 us at T = 512).
constexpr int kMoeNSmall = 128;
constexpr long long kSmallExpertBytes = 64ll << 20;
constexpr int kRouterTile = 16;      // tokens per router tile (router and permute tasks)
constexpr int kCombineTile = 16;     // most tokens per combine task
constexpr int kMoeSplitRowsCap = 512;  // split the down projection only up to T*k rows
constexpr int kGuSplitMax = 8;       // most K chunks of a gate/up tile (small batches)
constexpr int kGuRowsCap = 128;      // K chunks x T*k rows of gate/up partials at most

// split-K GEMM and MLP chain: up to 256 token rows per tile
constexpr int kWideNMax = 256;
constexpr int kMaxLayers = 4;        // MoE layers chained in one launch
constexpr int kLayerShift = 28;      // a task's layer, in the type word

// ---------------------------------------------------------------- workspace header

// The first 256 bytes of every workspace.  Everything but the sticky status
// word is returned to zero by the last CTA of each launch.
struct EtHeader {
    int32_t status_code;    // sticky first device error (et_status_code)
    int32_t status_detail;  // where it happened
    int32_t abort;          // non-zero: every bounded wait gives up
    int32_t exit_count;     // CTAs that left the task loop
    int32_t q_head;         // next task index to pop (dynamic queue)
    int32_t q_ready;        // the scan task has published the queue
    int32_t q_total;        // number of published queue entries
    int32_t total_mt;       // expert row tiles this call (published by the scan)
    int32_t ev_router;      // router tiles done
    int32_t ev_perm;        // permute tiles done
    int32_t ev_ydone;       // expert output tiles complete
    int32_t ev_norm;        // RMSNorm tasks done (MLP chain)
    int32_t split;          // split of the down projection chosen this call
    int32_t gu_split;       // K chunks of a gate/up tile chosen this call
    int32_t ev_sdone;       // shared-expert output tiles complete (fused block)
    int32_t q_wide;         // the down tiles are 256 columns wide this call
    int32_t reserved[48];
};
static_assert(sizeof(EtHeader) == 256, "header is 256 bytes");

constexpr int kHeaderBytes = 256;

// detail codes: where a wait ran out (low byte) and the CTA (upper bits)
enum WaitWhere {
    kWhereEmpty = 1,
    kWhereFull = 2,
    kWhereAcc = 3,
    kWhereQueue = 4,
    kWhereRouter = 5,
    kWherePerm = 6,
    kWhereH = 7,
    kWhereY = 8,
    kWhereNorm = 9,
    kWhereBoundsT = 10,
    kWhereStage = 11,
    kWhereInput = 12
};

// Task descriptor of the dynamic queue: {type, a, b, c}
enum TaskType { kTaskExit = 0, kTaskRouter = 1, kTaskScan = 2, kTaskPermute = 3,
                kTaskGateUp = 4, kTaskDown = 5, kTaskCombine = 6, kTaskNorm = 7,
                kTaskSplitK = 8, kTaskShGateUp = 9, kTaskShDown = 10, kTaskReduce = 11,
                kTaskNone = 15 /* producer only: nothing can be taken yet */ };

// ---------------------------------------------------------------- kernel argument blocks

struct MoeArgs {
    const bf16* x;        // [T, H]
    const bf16* wr;       // [H, E]
    const float* bias;    // [E] or null
    bf16* out;            // [T, H]
    int32_t* idx;         // [T_max, k]   (caller's buffer or workspace)
    float* gw;            // [T_max, k]
    int32_t* cnt;         // [E]
    int32_t* perm;        // [T_max * k]
    const int32_t* d_T;   // device token count or null
    int T_host, T_max, H, F, E, k;
    EtHeader* hdr;
    int32_t* ev_h;        // [mt_max * kSplitMax]
    int32_t* ev_y;        // [mt_max * (H/128)]
    int32_t* ev_tile;     // [r_max]: router expert chunks done per tile (self-resetting)
    float* logits;        // [T_max, E]: router logits when the experts are split in chunks
    int32_t* hist;        // [r_max * E]: per router tile expert histogram
    int32_t* base;        // [r_max * E]: first permuted row of each (tile, expert)
    int32_t* off;         // [E + 1]
    int32_t* pos;         // [T_max * k]: permuted row of (t, j)
    int4* g_info;         // [mt_max]: row tile g's {expert, first permuted row, rows, UMMA N}
    int4* e_tile;         // [E]: expert e's {first row tile, UMMA N, first permuted row, 0}
    int32_t* gpos;        // [T_max * k]: row tile of the permuted row of (t, j)
    int32_t* ev_gdone;    // [mt_max]: 128-column output tiles of row tile g complete
    bf16* xp;             // [T_max*k, H]: x rows in permuted order
    bf16* h;              // [T_max*k, F]
    bf16* y;              // [T_max*k, H]
    float* partial;       // [kSplitMax, split_rows_cap, H]
    float* gu_part;       // [2][gu_cap, F]: gate then up fp32 partials of K-split tiles
    int32_t* ev_gu;       // [mt_max * F/128]: K chunks done per gate/up tile (self-resetting)
    int gu_cap;           // rows of each gu_part half
    int mt_max, split_rows_cap, r_max;
    int split_mask;       // down splits d in [2, 8] that divide F/128 into chunks of >= 4 k-blocks (bit d)
    int kc_mask;          // gate/up K splits kc in {2, 4, 8} that divide H/64 into >= 8 k-blocks (bit kc)
    int wr_box;           // router-weight TMA box height (0: the weight is read in place)
    int b_wide;           // the 64-row activation maps are valid (enough rows)
    int num_ctas;
    // fused MoE block (gamma != null): x_hat = RMSNorm(x) * gamma routes and feeds
    // the experts; a shared SwiGLU expert (Fs > 0) and the residual join the combine
    const bf16* gamma;    // [H] or null (plain layer)
    float eps;
    int Fs;               // shared expert width (multiple of 128) or 0
    bf16* xn;             // [T_max, H]: x_hat
    bf16* hs;             // [T_max, Fs]: shared expert h
    bf16* ys;             // [T_max, H]: shared expert output
    int32_t* ev_hs;       // [mts_max * kSplitMax]: shared h tiles done per F-chunk
    int32_t* ev_ys;       // [mts_max * H/128]: shared split partials (self-resetting)
    float* partial_s;     // [kSplitMax, split_rows_cap, H]
    int mts_max;
    // chained layers: this layer's input is the previous layer's output
    const int32_t* ev_in;  // [r_max] previous layer's rows written per 16-token tile, or null
    int32_t* ev_tok;       // [r_max] this layer's rows written per 16-token tile, or null (last layer)
    uint64_t* trace;      // optional per-task trace (see et_opts)
    int trace_cap;
    uint64_t timeout_ns;
    int fault_mode, fault_arg;
};

struct SplitKArgs {
    bf16* Y;              // [M, N]
    const int32_t* d_M;
    int M_host, M_max, N, K, split;
    EtHeader* hdr;
    int32_t* ev;          // [ceil(M_max/256) * N/128], self-resetting
    float* partial;       // [split, M_max, N]
    int b_wide;
    int num_ctas;
    uint64_t timeout_ns;
    int fault_mode, fault_arg;
    uint64_t* trace;      // optional per-task trace (see et_opts)
    int trace_cap;
};

struct MlpArgs {
    const bf16* x;        // [B, H]
    const bf16* gamma;    // [H]
    float eps;
    bf16* out;            // [B, H]
    const int32_t* d_B;
    int B_host, B_max, H, F;
    EtHeader* hdr;
    bf16* xhat;           // [B_max, H]
    bf16* h;              // [B_max, F]
    int32_t* ev_h;        // [mt_max * kMlpSplitMax]
    int32_t* ev_y;        // [mt_max * H/128], self-resetting
    float* partial;       // [kMlpSplitMax, B_max, H]
    float* gu_part;       // [2][gu_cap, F]: gate then up fp32 partials of K-split tiles
    int32_t* ev_gu;       // [mt_max * F/128]: K chunks done per gate/up tile (self-resetting)
    int gu_cap;           // rows of each gu_part half (K chunks x batch rows)
    int mt_max;
    int b_wide;
    int num_ctas;
    uint64_t timeout_ns;
    int fault_mode, fault_arg;
    uint64_t* trace;      // optional per-task trace (see et_opts)
    int trace_cap;
};
constexpr int kMlpGuRowsCap = 256;   // MLP: K chunks x B rows of gate/up partials at most
constexpr int kMlpSplitMax = 16;     // MLP: largest split of the down projection

}  // namespace et
