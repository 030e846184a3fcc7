// etmoe_api.cu -- the C ABI of libetmoe.so: argument checks, workspace
// carve-up, TMA tensor maps, and one cooperative launch per call.  No call
// here allocates device memory or synchronises, except et_status.
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>
#include <string>

#include "et_gemm.cuh"

namespace et {
cudaError_t launch_moe(const MoeArgs*, const CUtensorMap*, int, int, int, cudaStream_t);
cudaError_t prepare_moe(int);
int moe_smem_bytes();
int moe_ring_bytes();
cudaError_t launch_splitk(const SplitKArgs&, const CUtensorMap*, int, int, cudaStream_t);
cudaError_t prepare_splitk(int);
int splitk_smem_bytes();
cudaError_t launch_splitk_clc(const SplitKArgs&, const CUtensorMap*, int, int, cudaStream_t);
cudaError_t prepare_splitk_clc(int);
int splitk_clc_smem_bytes();
cudaError_t launch_mlp(const MlpArgs&, const CUtensorMap*, int, int, cudaStream_t);
cudaError_t prepare_mlp(int);
int mlp_smem_bytes();
}  // namespace et

using namespace et;

namespace {

thread_local std::string g_last_error;

int fail(int code, const std::string& msg) {
    g_last_error = msg;
    return code;
}

int fail_cuda(cudaError_t e, const char* what) {
    return fail(ET_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    int sms = 0;
    bool moe = false, splitk = false, splitk_clc = false, mlp = false;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

template <class T>
bool aligned(const void* p, size_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Per-device one-time set-up: SM count, kernel attributes, the driver's
// tensor-map encoder (fetched through the runtime, so the library does not
// link libcuda and loads on machines without a GPU).
int device_state(DeviceState** out, int* dev_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(ET_ERR_CUDA, "device index out of range");
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState& st = g_dev[dev];
    if (!st.ready) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (major != 10 || minor != 3)
            return fail(ET_ERR_UNSUPPORTED, "libetmoe is built for sm_103a (GB300) only; device is sm_" +
                                                std::to_string(major) + std::to_string(minor));
        e = cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute(SM count)");
        if (!g_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
                return fail(ET_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        st.ready = true;
    }
    *out = &st;
    if (dev_out) *dev_out = dev;
    return ET_OK;
}

// Row-major bf16 matrix [rows, cols] as a 2-D tensor map with 64-column,
// box_rows-row boxes and the 128-byte swizzle (one swizzle row = 64 bf16).
int make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
             const char* what) {
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kBlockK), box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(ET_ERR_CUDA, std::string("cuTensorMapEncodeTiled failed for ") + what +
                                     " (code " + std::to_string(static_cast<int>(r)) + ")");
    return ET_OK;
}

// Row-major bf16 [rows, cols] without swizzle, box {box_cols, box_rows}
// (box_cols * 2 a multiple of 16 bytes, cols * 2 too).
int make_map_plain(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                   uint32_t box_cols, uint32_t box_rows, const char* what) {
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return fail(ET_ERR_CUDA, std::string("cuTensorMapEncodeTiled failed for ") + what +
                                     " (code " + std::to_string(static_cast<int>(r)) + ")");
    return ET_OK;
}

uint64_t timeout_ns_of(const et_opts* o) {
    const uint32_t us = (o && o->timeout_us) ? o->timeout_us : 200000u;
    return static_cast<uint64_t>(us) * 1000ull;
}

struct Carve {
    size_t off = kHeaderBytes;
    size_t take(size_t bytes, size_t align = 256) {
        off = round_up(off, align);
        const size_t r = off;
        off += round_up(bytes, 16);
        return r;
    }
};

// ---------------------------------------------------------------- MoE layout

struct MoeLayout {
    int Tk, r_max, mt_max, split_cap, gu_cap, mts_max;
    size_t ev_h, ev_y, ev_tile, ev_gu, logits, hist, base, idx, gw, cnt, off, pos, perm, g_info,
        e_tile, gpos, ev_gdone, xp, h, y, partial, gu_part;
    size_t xn, hs, ys, ev_hs, ev_ys, partial_s;  // fused block only (block == true)
    size_t ev_tok;                               // rows released per 16-token tile (chains)
    size_t total;
};

// block: the fused MoE block's extra regions (x_hat; with Fs > 0 the shared
// expert's h, y, counters and split partials).
MoeLayout moe_layout(int T_max, int H, int F, int E, int k, bool block = false, int Fs = 0) {
    MoeLayout L{};
    L.Tk = T_max * k;
    L.r_max = ceil_div(T_max, kRouterTile);
    L.mt_max = ceil_div(L.Tk, kMoeNSmall / 2) + E;  // row tiles at the smallest cap
    const int FT = F / kTileM, HT = H / kTileM;
    L.mts_max = (block && Fs > 0) ? ceil_div(T_max, kWideNMax) : 0;
    L.split_cap = L.Tk < kMoeSplitRowsCap ? L.Tk : kMoeSplitRowsCap;
    L.gu_cap = L.Tk * kGuSplitMax < kGuRowsCap ? L.Tk * kGuSplitMax : kGuRowsCap;
    Carve c;
    L.ev_h = c.take(sizeof(int) * L.mt_max * kSplitMax);
    L.ev_y = c.take(sizeof(int) * L.mt_max * HT);
    L.ev_tile = c.take(sizeof(int) * L.r_max);
    L.ev_gu = c.take(sizeof(int) * L.mt_max * FT);
    L.logits = c.take(sizeof(float) * static_cast<size_t>(T_max) * E);
    L.hist = c.take(sizeof(int) * L.r_max * E);
    L.base = c.take(sizeof(int) * L.r_max * E);
    L.idx = c.take(sizeof(int) * L.Tk);
    L.gw = c.take(sizeof(float) * L.Tk);
    L.cnt = c.take(sizeof(int) * E);
    L.off = c.take(sizeof(int) * (E + 1));
    L.pos = c.take(sizeof(int) * L.Tk);
    L.perm = c.take(sizeof(int) * L.Tk);
    L.g_info = c.take(sizeof(int4) * L.mt_max);
    L.e_tile = c.take(sizeof(int4) * E);
    L.gpos = c.take(sizeof(int) * L.Tk);
    L.ev_gdone = c.take(sizeof(int) * L.mt_max);
    L.xp = c.take(sizeof(uint16_t) * static_cast<size_t>(L.Tk) * H, 1024);
    L.h = c.take(sizeof(uint16_t) * static_cast<size_t>(L.Tk) * F, 1024);
    L.y = c.take(sizeof(uint16_t) * static_cast<size_t>(L.Tk) * H, 1024);
    L.partial = c.take(sizeof(float) * static_cast<size_t>(kSplitMax) * L.split_cap * H, 1024);
    L.gu_part = c.take(sizeof(float) * 2 * static_cast<size_t>(L.gu_cap) * F, 1024);
    L.ev_tok = c.take(sizeof(int) * L.r_max);
    if (block) {
        L.xn = c.take(sizeof(uint16_t) * static_cast<size_t>(T_max) * H, 1024);
        if (Fs > 0) {
            L.ev_hs = c.take(sizeof(int) * L.mts_max * kSplitMax);
            L.ev_ys = c.take(sizeof(int) * L.mts_max * HT);
            L.hs = c.take(sizeof(uint16_t) * static_cast<size_t>(T_max) * Fs, 1024);
            L.ys = c.take(sizeof(uint16_t) * static_cast<size_t>(T_max) * H, 1024);
            L.partial_s = c.take(sizeof(float) * static_cast<size_t>(kSplitMax) * L.split_cap * H, 1024);
        }
    }
    L.total = round_up(c.off, 256);
    return L;
}

bool moe_shape_ok(int T_max, int H, int F, int E, int k, std::string* why) {
    if (T_max < 1 || T_max > 65536) { *why = "T_max must be in [1, 65536]"; return false; }
    if (H < 128 || H % 128 || F < 128 || F % 128) { *why = "H and F must be positive multiples of 128"; return false; }
    if (H > 65536 || F > 65536) { *why = "H and F must be <= 65536"; return false; }
    if (E < 1 || E > 256) { *why = "E must be in [1, 256]"; return false; }
    if (k < 1 || k > 8 || k > E) { *why = "k must be in [1, min(E, 8)]"; return false; }
    if (static_cast<long long>(E) * F >= (1ll << 31) || static_cast<long long>(E) * H >= (1ll << 31)) {
        *why = "E*F and E*H must fit in int32"; return false;
    }
    if (static_cast<long long>(k) * H * 2 > moe_ring_bytes()) {  // one token's k rows are staged at once
        *why = "k*H*2 bytes must fit in the stage ring (" + std::to_string(moe_ring_bytes()) + ")";
        return false;
    }
    return true;
}

// The fused block stages k + 2 rows per token in the combine (the k expert
// rows, the residual and the shared expert's row).
bool block_shape_ok(int T_max, int H, int F, int E, int k, int Fs, std::string* why) {
    if (!moe_shape_ok(T_max, H, F, E, k, why)) return false;
    if (Fs < 0 || Fs % 128 || Fs > 65536) {
        *why = "Fs must be 0 or a positive multiple of 128 (<= 65536)"; return false;
    }
    const long long rows = k + 1 + (Fs > 0 ? 1 : 0);
    if (rows * H * 2 > moe_ring_bytes()) {
        *why = "(k+2)*H*2 bytes must fit in the stage ring (" + std::to_string(moe_ring_bytes()) + ")";
        return false;
    }
    return true;
}

// Fused-block inputs of the shared launch path (on == false: the plain layer).
struct BlockIn {
    bool on;
    const void* gamma;
    float eps;
    int Fs;
    const void *ws_gate, *ws_up, *ws_down;
    void* x_hat;
};

// ---------------------------------------------------------------- split-K layout

struct SplitKLayout {
    size_t ev, partial, total;
};

SplitKLayout splitk_layout(int M_max, int N, int K, int split) {
    (void)K;
    SplitKLayout L{};
    Carve c;
    L.ev = c.take(sizeof(int) * static_cast<size_t>(ceil_div(M_max, kWideNMax)) * (N / kTileM));
    L.partial = c.take(sizeof(float) * static_cast<size_t>(split > 1 ? split : 0) * M_max * N, 1024);
    L.total = round_up(c.off, 256);
    return L;
}

// ---------------------------------------------------------------- MLP layout

struct MlpLayout {
    int mt_max, gu_cap;
    size_t xhat, h, ev_h, ev_y, ev_gu, partial, gu_part, total;
};

MlpLayout mlp_layout(int B_max, int H, int F) {
    MlpLayout L{};
    L.mt_max = ceil_div(B_max, kWideNMax);
    Carve c;
    L.ev_h = c.take(sizeof(int) * L.mt_max * kMlpSplitMax);
    L.ev_y = c.take(sizeof(int) * L.mt_max * (H / kTileM));
    L.xhat = c.take(sizeof(uint16_t) * static_cast<size_t>(B_max) * H, 1024);
    L.h = c.take(sizeof(uint16_t) * static_cast<size_t>(B_max) * F, 1024);
    L.partial = c.take(sizeof(float) * static_cast<size_t>(kMlpSplitMax) * B_max * H, 1024);
    L.gu_cap = B_max * kGuSplitMax < kMlpGuRowsCap ? B_max * kGuSplitMax : kMlpGuRowsCap;
    L.ev_gu = c.take(sizeof(int) * L.mt_max * (F / kTileM));
    L.gu_part = c.take(sizeof(float) * 2 * static_cast<size_t>(L.gu_cap) * F, 1024);
    L.total = round_up(c.off, 256);
    return L;
}

int check_ws(void* ws, size_t have, size_t need) {
    if (!ws) return fail(ET_ERR_WORKSPACE, "workspace is NULL");
    if (!aligned<void>(ws, 256)) return fail(ET_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (have < need)
        return fail(ET_ERR_WORKSPACE, "workspace too small: need " + std::to_string(need) +
                                          " bytes, got " + std::to_string(have));
    return ET_OK;
}

}  // namespace

extern "C" {

int et_version(void) { return 100; }

const char* et_last_error_string(void) { return g_last_error.c_str(); }

size_t et_moe_workspace_bytes(int T_max, int H, int F, int E, int k) {
    std::string why;
    if (!moe_shape_ok(T_max, H, F, E, k, &why)) return 0;
    return moe_layout(T_max, H, F, E, k).total;
}

}  // extern "C"

namespace {

// One layer of a launch as the host sees it (a plain layer, or a fused block
// when b.on).
struct LayerIn {
    BlockIn b;
    const void* w_router;
    const float* bias;
    const void *w_gate, *w_up, *w_down;
    void* out;
    int32_t* topk_idx;
    float* topk_w;
    int32_t* expert_counts;
    int32_t* perm;
};

// Workspace of a launch: one region per layer, each [header | layout].
size_t chain_bytes(const LayerIn* layers, int nl, int T_max, int H, int F, int E, int k,
                   size_t* offs) {
    size_t off = 0;
    for (int l = 0; l < nl; ++l) {
        if (offs) offs[l] = off;
        off += moe_layout(T_max, H, F, E, k, layers[l].b.on, layers[l].b.Fs).total;
    }
    return off;
}

// Every MoE entry point ends here: nl chained layers (shapes validated by the
// caller), layer l + 1 reading layer l's output, in one launch.
int moe_run(const void* x, const LayerIn* layers, int nl, int T, const int32_t* d_T, int T_max,
            int H, int F, int E, int k, void* workspace, size_t workspace_bytes,
            const et_opts* opts, void* stream) {
    if (nl < 1 || nl > kMaxLayers) return fail(ET_ERR_INVALID, "1 to 4 layers per launch");
    if (!x) return fail(ET_ERR_INVALID, "x must be non-NULL");
    if (!aligned<void>(x, 16)) return fail(ET_ERR_INVALID, "tensors must be 16-byte aligned");
    for (int l = 0; l < nl; ++l) {
        const LayerIn& li = layers[l];
        if (!li.w_router || !li.w_gate || !li.w_up || !li.w_down || !li.out)
            return fail(ET_ERR_INVALID, "w_router, w_gate, w_up, w_down and out must be non-NULL");
        const void* need16[] = {li.w_router, li.w_gate, li.w_up, li.w_down, li.out};
        for (const void* q : need16)
            if (!aligned<void>(q, 16)) return fail(ET_ERR_INVALID, "tensors must be 16-byte aligned");
    }
    if (!d_T && (T < 0 || T > T_max)) return fail(ET_ERR_INVALID, "T must be in [0, T_max]");
    size_t offs[kMaxLayers];
    const size_t total = chain_bytes(layers, nl, T_max, H, F, E, k, offs);
    int rc = check_ws(workspace, workspace_bytes, total);
    if (rc) return rc;
    if (!d_T && T == 0) return ET_OK;

    DeviceState* st = nullptr;
    if ((rc = device_state(&st, nullptr))) return rc;
    const int smem = moe_smem_bytes();
    if (!st->moe) {
        cudaError_t e = prepare_moe(smem);
        if (e != cudaSuccess) return fail_cuda(e, "cudaFuncSetAttribute(moe)");
        st->moe = true;
    }
    MoeArgs args[kMaxLayers];
    constexpr int kMaps = 14;  // tensor maps a layer (the kernel's MoeLayerMaps)
    CUtensorMap maps[kMaps * kMaxLayers];
    for (int l = 0; l < nl; ++l) {
        const LayerIn& li = layers[l];
        const BlockIn& b = li.b;
        const MoeLayout L = moe_layout(T_max, H, F, E, k, b.on, b.Fs);
        uint8_t* ws = static_cast<uint8_t*>(workspace) + offs[l];
        MoeArgs& a = args[l];
        a = MoeArgs{};
        a.x = static_cast<const bf16*>(l == 0 ? x : layers[l - 1].out);
        a.wr = static_cast<const bf16*>(li.w_router);
        a.bias = li.bias;
        a.out = static_cast<bf16*>(li.out);
        a.idx = li.topk_idx ? li.topk_idx : reinterpret_cast<int32_t*>(ws + L.idx);
        a.gw = li.topk_w ? li.topk_w : reinterpret_cast<float*>(ws + L.gw);
        a.cnt = li.expert_counts ? li.expert_counts : reinterpret_cast<int32_t*>(ws + L.cnt);
        a.perm = li.perm ? li.perm : reinterpret_cast<int32_t*>(ws + L.perm);
        a.d_T = d_T;
        a.T_host = T;
        a.T_max = T_max;
        a.H = H;
        a.F = F;
        a.E = E;
        a.k = k;
        a.hdr = reinterpret_cast<EtHeader*>(ws);
        a.ev_h = reinterpret_cast<int32_t*>(ws + L.ev_h);
        a.ev_y = reinterpret_cast<int32_t*>(ws + L.ev_y);
        a.ev_tile = reinterpret_cast<int32_t*>(ws + L.ev_tile);
        a.logits = reinterpret_cast<float*>(ws + L.logits);
        a.hist = reinterpret_cast<int32_t*>(ws + L.hist);
        a.base = reinterpret_cast<int32_t*>(ws + L.base);
        a.off = reinterpret_cast<int32_t*>(ws + L.off);
        a.pos = reinterpret_cast<int32_t*>(ws + L.pos);
        a.g_info = reinterpret_cast<int4*>(ws + L.g_info);
        a.e_tile = reinterpret_cast<int4*>(ws + L.e_tile);
        a.gpos = reinterpret_cast<int32_t*>(ws + L.gpos);
        a.ev_gdone = reinterpret_cast<int32_t*>(ws + L.ev_gdone);
        a.xp = reinterpret_cast<bf16*>(ws + L.xp);
        a.h = reinterpret_cast<bf16*>(ws + L.h);
        a.y = reinterpret_cast<bf16*>(ws + L.y);
        a.partial = reinterpret_cast<float*>(ws + L.partial);
        a.gu_part = reinterpret_cast<float*>(ws + L.gu_part);
        a.ev_gu = reinterpret_cast<int32_t*>(ws + L.ev_gu);
        a.gu_cap = L.gu_cap;
        a.mt_max = L.mt_max;
        a.split_rows_cap = L.split_cap;
        a.r_max = L.r_max;
        a.wr_box = E % 8 == 0 ? (H % 256 == 0 ? 256 : 128) : 0;
        a.split_mask = 0;
        for (int d = 2; d <= kSplitMax; ++d)
            if ((F / kTileM) % d == 0 && F / kBlockK / d >= 4) a.split_mask |= 1 << d;
        a.kc_mask = 0;
        for (int kc = 2; kc <= kGuSplitMax; kc *= 2)
            if ((H / kBlockK) % kc == 0 && H / kBlockK / kc >= 8) a.kc_mask |= 1 << kc;
        a.num_ctas = st->sms;
        a.timeout_ns = timeout_ns_of(opts);
        a.fault_mode = (opts && l == 0) ? opts->fault_mode : 0;
        a.fault_arg = (opts && l == 0) ? opts->fault_arg : 0;
        a.trace = (opts && opts->trace && opts->trace_cap) ? static_cast<uint64_t*>(opts->trace)
                                                           : nullptr;
        a.trace_cap = opts ? static_cast<int>(opts->trace_cap) : 0;
        a.ev_in = l > 0 ? args[l - 1].ev_tok : nullptr;
        a.ev_tok = l + 1 < nl ? reinterpret_cast<int32_t*>(ws + L.ev_tok) : nullptr;
        if (b.on) {
            a.gamma = static_cast<const bf16*>(b.gamma);
            a.eps = b.eps;
            a.Fs = b.Fs;
            a.xn = b.x_hat ? static_cast<bf16*>(b.x_hat) : reinterpret_cast<bf16*>(ws + L.xn);
            if (b.Fs > 0) {
                a.hs = reinterpret_cast<bf16*>(ws + L.hs);
                a.ys = reinterpret_cast<bf16*>(ws + L.ys);
                a.ev_hs = reinterpret_cast<int32_t*>(ws + L.ev_hs);
                a.ev_ys = reinterpret_cast<int32_t*>(ws + L.ev_ys);
                a.partial_s = reinterpret_cast<float*>(ws + L.partial_s);
                a.mts_max = L.mts_max;
            }
        }

        CUtensorMap* mp = maps + kMaps * l;
        const uint64_t EF = static_cast<uint64_t>(E) * F, EH = static_cast<uint64_t>(E) * H;
        if ((rc = make_map(&mp[0], li.w_gate, EF, H, kTileM, "w_gate"))) return rc;
        if ((rc = make_map(&mp[1], li.w_up, EF, H, kTileM, "w_up"))) return rc;
        if ((rc = make_map(&mp[2], li.w_down, EH, F, kTileM, "w_down"))) return rc;
        if ((rc = make_map(&mp[3], a.xp, L.Tk, H, kBBoxRows, "permuted x"))) return rc;
        if ((rc = make_map(&mp[4], a.h, L.Tk, F, kBBoxRows, "h"))) return rc;
        if (a.wr_box) {
            if ((rc = make_map_plain(&mp[5], li.w_router, H, E, 8, a.wr_box, "w_router"))) return rc;
        } else {
            mp[5] = mp[0];  // unused: the router weight is read in place
        }
        a.b_wide = L.Tk >= kBBoxRowsWide ? 1 : 0;
        if (a.b_wide) {
            if ((rc = make_map(&mp[6], a.xp, L.Tk, H, kBBoxRowsWide, "permuted x"))) return rc;
            if ((rc = make_map(&mp[7], a.h, L.Tk, F, kBBoxRowsWide, "h"))) return rc;
        } else {
            mp[6] = mp[3];
            mp[7] = mp[4];
        }
        for (int i = 8; i < 13; ++i) mp[i] = mp[0];  // unused unless the shared expert runs
        if (b.on && b.Fs > 0) {
            const uint64_t Fs = static_cast<uint64_t>(b.Fs);
            if ((rc = make_map(&mp[8], b.ws_gate, Fs, H, kTileM, "ws_gate"))) return rc;
            if ((rc = make_map(&mp[9], b.ws_up, Fs, H, kTileM, "ws_up"))) return rc;
            if ((rc = make_map(&mp[10], b.ws_down, H, Fs, kTileM, "ws_down"))) return rc;
            if ((rc = make_map(&mp[11], a.xn, T_max, H, kBBoxRows, "x_hat"))) return rc;
            if ((rc = make_map(&mp[12], a.hs, T_max, Fs, kBBoxRows, "shared h"))) return rc;
        }
        // the router's input rows (x_hat in a fused block), 16-row boxes
        if ((rc = make_map(&mp[13], b.on ? static_cast<const void*>(a.xn) : static_cast<const void*>(a.x),
                           T_max, H, kBBoxRows, "router input")))
            return rc;
    }
    cudaError_t e = launch_moe(args, maps, nl, st->sms, smem, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e, "launch of the MoE megakernel");
    return ET_OK;
}

}  // namespace

extern "C" {

int et_moe_layer(const void* x, const void* w_router, const float* router_bias, const void* w_gate,
                 const void* w_up, const void* w_down, void* out, int32_t* topk_idx, float* topk_w,
                 int32_t* expert_counts, int32_t* perm, int T, const int32_t* d_T, int T_max, int H,
                 int F, int E, int k, void* workspace, size_t workspace_bytes, const et_opts* opts,
                 void* stream) {
    g_last_error.clear();
    std::string why;
    if (!moe_shape_ok(T_max, H, F, E, k, &why)) return fail(ET_ERR_UNSUPPORTED, why);
    LayerIn li{BlockIn{}, w_router, router_bias, w_gate, w_up, w_down, out, topk_idx, topk_w,
               expert_counts, perm};
    return moe_run(x, &li, 1, T, d_T, T_max, H, F, E, k, workspace, workspace_bytes, opts, stream);
}

size_t et_moe_block_workspace_bytes(int T_max, int H, int F, int E, int k, int Fs) {
    std::string why;
    if (!block_shape_ok(T_max, H, F, E, k, Fs, &why)) return 0;
    return moe_layout(T_max, H, F, E, k, true, Fs).total;
}

int et_moe_block(const void* x, const void* gamma, float eps, const void* w_router,
                 const float* router_bias, const void* w_gate, const void* w_up, const void* w_down,
                 const void* ws_gate, const void* ws_up, const void* ws_down, int Fs, void* out,
                 void* x_hat, int32_t* topk_idx, float* topk_w, int32_t* expert_counts,
                 int32_t* perm, int T, const int32_t* d_T, int T_max, int H, int F, int E, int k,
                 void* workspace, size_t workspace_bytes, const et_opts* opts, void* stream) {
    g_last_error.clear();
    std::string why;
    if (!block_shape_ok(T_max, H, F, E, k, Fs, &why)) return fail(ET_ERR_UNSUPPORTED, why);
    if (!gamma) return fail(ET_ERR_INVALID, "gamma must be non-NULL");
    if (!(eps > 0.0f) || !std::isfinite(eps)) return fail(ET_ERR_INVALID, "eps must be finite and > 0");
    if (Fs > 0 && (!ws_gate || !ws_up || !ws_down))
        return fail(ET_ERR_INVALID, "ws_gate, ws_up and ws_down must be non-NULL when Fs > 0");
    const void* need16[] = {gamma, ws_gate, ws_up, ws_down, x_hat};
    for (const void* q : need16)
        if (q && !aligned<void>(q, 16)) return fail(ET_ERR_INVALID, "tensors must be 16-byte aligned");
    LayerIn li{BlockIn{true, gamma, eps, Fs, ws_gate, ws_up, ws_down, x_hat}, w_router,
               router_bias, w_gate, w_up, w_down, out, topk_idx, topk_w, expert_counts, perm};
    return moe_run(x, &li, 1, T, d_T, T_max, H, F, E, k, workspace, workspace_bytes, opts, stream);
}

}  // extern "C"

namespace {

// Validate a chain's descriptors and turn them into launch layers.
int chain_layers(int n_layers, const et_moe_layer_desc* d, int T_max, int H, int F, int E, int k,
                 LayerIn* out, std::string* why) {
    if (n_layers < 1 || n_layers > kMaxLayers || !d) {
        *why = "n_layers must be in [1, 4] and layers non-NULL";
        return ET_ERR_INVALID;
    }
    for (int l = 0; l < n_layers; ++l) {
        const et_moe_layer_desc& q = d[l];
        const bool block = q.gamma != nullptr;
        if (block ? !block_shape_ok(T_max, H, F, E, k, q.Fs, why)
                  : !moe_shape_ok(T_max, H, F, E, k, why))
            return ET_ERR_UNSUPPORTED;
        if (!block && q.Fs != 0) {
            *why = "a layer without gamma has no shared expert (Fs must be 0)";
            return ET_ERR_INVALID;
        }
        if (block) {
            if (!(q.eps > 0.0f) || !std::isfinite(q.eps)) {
                *why = "eps must be finite and > 0";
                return ET_ERR_INVALID;
            }
            if (q.Fs > 0 && (!q.ws_gate || !q.ws_up || !q.ws_down)) {
                *why = "ws_gate, ws_up and ws_down must be non-NULL when Fs > 0";
                return ET_ERR_INVALID;
            }
            const void* need16[] = {q.gamma, q.ws_gate, q.ws_up, q.ws_down, q.x_hat};
            for (const void* v : need16)
                if (v && !aligned<void>(v, 16)) {
                    *why = "tensors must be 16-byte aligned";
                    return ET_ERR_INVALID;
                }
        }
        out[l] = LayerIn{BlockIn{block, q.gamma, q.eps, block ? q.Fs : 0, q.ws_gate, q.ws_up,
                                 q.ws_down, q.x_hat},
                         q.w_router, q.router_bias, q.w_gate, q.w_up, q.w_down, q.out,
                         q.topk_idx, q.topk_w, q.expert_counts, q.perm};
    }
    return ET_OK;
}

}  // namespace

extern "C" {

size_t et_moe_chain_workspace_bytes(int n_layers, const et_moe_layer_desc* layers, int T_max,
                                    int H, int F, int E, int k) {
    LayerIn li[kMaxLayers];
    std::string why;
    if (chain_layers(n_layers, layers, T_max, H, F, E, k, li, &why) != ET_OK) return 0;
    return chain_bytes(li, n_layers, T_max, H, F, E, k, nullptr);
}

int et_moe_chain(int n_layers, const et_moe_layer_desc* layers, const void* x, int T,
                 const int32_t* d_T, int T_max, int H, int F, int E, int k, void* workspace,
                 size_t workspace_bytes, const et_opts* opts, void* stream) {
    g_last_error.clear();
    LayerIn li[kMaxLayers];
    std::string why;
    const int rc = chain_layers(n_layers, layers, T_max, H, F, E, k, li, &why);
    if (rc != ET_OK) return fail(rc, why);
    return moe_run(x, li, n_layers, T, d_T, T_max, H, F, E, k, workspace, workspace_bytes, opts,
                   stream);
}

size_t et_splitk_workspace_bytes(int M_max, int N, int K, int split) {
    if (M_max < 1 || N < 128 || N % 128 || split < 1 || split > 16 || K < 64 || K % (64 * split))
        return 0;
    return splitk_layout(M_max, N, K, split).total;
}

}  // extern "C"

namespace {

// The split-K GEMM: the static, cooperative schedule (clc == false) or the
// Cluster Launch Control work queue (clc == true).
int splitk_run(const void* X, const void* Wt, void* Y, int M, const int32_t* d_M, int M_max, int N,
               int K, int split, void* workspace, size_t workspace_bytes, const et_opts* opts,
               void* stream, bool clc) {
    if (M_max < 1 || M_max > (1 << 20)) return fail(ET_ERR_INVALID, "M_max must be in [1, 2^20]");
    if (N < 128 || N % 128 || N > (1 << 20))
        return fail(ET_ERR_UNSUPPORTED, "N must be a positive multiple of 128");
    if (split < 1 || split > 16) return fail(ET_ERR_UNSUPPORTED, "split must be in [1, 16]");
    if (K < 64 || K % (64 * split) || K > (1 << 22))
        return fail(ET_ERR_UNSUPPORTED, "K must be a positive multiple of 64*split");
    if (!X || !Wt || !Y) return fail(ET_ERR_INVALID, "X, Wt and Y must be non-NULL");
    if (!aligned<void>(X, 16) || !aligned<void>(Wt, 16) || !aligned<void>(Y, 16))
        return fail(ET_ERR_INVALID, "tensors must be 16-byte aligned");
    if (!d_M && (M < 0 || M > M_max)) return fail(ET_ERR_INVALID, "M must be in [0, M_max]");
    const SplitKLayout L = splitk_layout(M_max, N, K, split);
    int rc = check_ws(workspace, workspace_bytes, L.total);
    if (rc) return rc;
    if (!d_M && M == 0) return ET_OK;
    DeviceState* st = nullptr;
    if ((rc = device_state(&st, nullptr))) return rc;
    const int smem = clc ? splitk_clc_smem_bytes() : splitk_smem_bytes();
    bool& prepared = clc ? st->splitk_clc : st->splitk;
    if (!prepared) {
        cudaError_t e = clc ? prepare_splitk_clc(smem) : prepare_splitk(smem);
        if (e != cudaSuccess) return fail_cuda(e, "cudaFuncSetAttribute(splitk)");
        prepared = true;
    }
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    SplitKArgs a{};
    a.Y = static_cast<bf16*>(Y);
    a.d_M = d_M;
    a.M_host = M;
    a.M_max = M_max;
    a.N = N;
    a.K = K;
    a.split = split;
    a.hdr = reinterpret_cast<EtHeader*>(ws);
    a.ev = reinterpret_cast<int32_t*>(ws + L.ev);
    a.partial = reinterpret_cast<float*>(ws + L.partial);
    a.num_ctas = st->sms;
    a.timeout_ns = timeout_ns_of(opts);
    a.fault_mode = opts ? opts->fault_mode : 0;
    a.fault_arg = opts ? opts->fault_arg : 0;
    a.trace = (opts && opts->trace && opts->trace_cap) ? static_cast<uint64_t*>(opts->trace) : nullptr;
    a.trace_cap = opts ? static_cast<int>(opts->trace_cap) : 0;
    CUtensorMap maps[3];
    if ((rc = make_map(&maps[0], Wt, N, K, kTileM, "Wt"))) return rc;
    if ((rc = make_map(&maps[1], X, M_max, K, kBBoxRows, "X"))) return rc;
    a.b_wide = M_max >= kBBoxRowsWide ? 1 : 0;
    if (a.b_wide) {
        if ((rc = make_map(&maps[2], X, M_max, K, kBBoxRowsWide, "X"))) return rc;
    } else {
        maps[2] = maps[1];
    }
    // the hardware queue's grid: one CTA per tile task of every M tile up to M_max
    const long long tasks = static_cast<long long>(ceil_div(M_max, kWideNMax)) * (N / kTileM) * split;
    cudaError_t e = clc ? launch_splitk_clc(a, maps, static_cast<int>(tasks), smem,
                                            static_cast<cudaStream_t>(stream))
                        : launch_splitk(a, maps, st->sms, smem, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e, "launch of the split-K kernel");
    return ET_OK;
}

}  // namespace

extern "C" {

int et_splitk_gemm(const void* X, const void* Wt, void* Y, int M, const int32_t* d_M, int M_max,
                   int N, int K, int split, void* workspace, size_t workspace_bytes,
                   const et_opts* opts, void* stream) {
    g_last_error.clear();
    return splitk_run(X, Wt, Y, M, d_M, M_max, N, K, split, workspace, workspace_bytes, opts,
                      stream, false);
}

int et_splitk_gemm_clc(const void* X, const void* Wt, void* Y, int M, const int32_t* d_M,
                       int M_max, int N, int K, int split, void* workspace,
                       size_t workspace_bytes, const et_opts* opts, void* stream) {
    g_last_error.clear();
    return splitk_run(X, Wt, Y, M, d_M, M_max, N, K, split, workspace, workspace_bytes, opts,
                      stream, true);
}

size_t et_mlp_workspace_bytes(int B_max, int H, int F) {
    if (B_max < 1 || B_max > 65536 || H < 128 || H % 128 || F < 128 || F % 128) return 0;
    return mlp_layout(B_max, H, F).total;
}

int et_mlp_chain(const void* x, const void* gamma, float eps, const void* w_gate, const void* w_up,
                 const void* w_down, void* out, int B, const int32_t* d_B, int B_max, int H, int F,
                 void* workspace, size_t workspace_bytes, const et_opts* opts, void* stream) {
    g_last_error.clear();
    if (B_max < 1 || B_max > 65536) return fail(ET_ERR_INVALID, "B_max must be in [1, 65536]");
    if (H < 128 || H % 128 || F < 128 || F % 128 || H > 65536 || F > 65536)
        return fail(ET_ERR_UNSUPPORTED, "H and F must be positive multiples of 128 (<= 65536)");
    if (!x || !gamma || !w_gate || !w_up || !w_down || !out)
        return fail(ET_ERR_INVALID, "x, gamma, w_gate, w_up, w_down and out must be non-NULL");
    const void* need16[] = {x, gamma, w_gate, w_up, w_down, out};
    for (const void* p : need16)
        if (!aligned<void>(p, 16)) return fail(ET_ERR_INVALID, "tensors must be 16-byte aligned");
    if (!(eps >= 0.0f)) return fail(ET_ERR_INVALID, "eps must be >= 0");
    if (!d_B && (B < 0 || B > B_max)) return fail(ET_ERR_INVALID, "B must be in [0, B_max]");
    const MlpLayout L = mlp_layout(B_max, H, F);
    int rc = check_ws(workspace, workspace_bytes, L.total);
    if (rc) return rc;
    if (!d_B && B == 0) return ET_OK;
    DeviceState* st = nullptr;
    if ((rc = device_state(&st, nullptr))) return rc;
    const int smem = mlp_smem_bytes();
    if (!st->mlp) {
        cudaError_t e = prepare_mlp(smem);
        if (e != cudaSuccess) return fail_cuda(e, "cudaFuncSetAttribute(mlp)");
        st->mlp = true;
    }
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    MlpArgs a{};
    a.x = static_cast<const bf16*>(x);
    a.gamma = static_cast<const bf16*>(gamma);
    a.eps = eps;
    a.out = static_cast<bf16*>(out);
    a.d_B = d_B;
    a.B_host = B;
    a.B_max = B_max;
    a.H = H;
    a.F = F;
    a.hdr = reinterpret_cast<EtHeader*>(ws);
    a.xhat = reinterpret_cast<bf16*>(ws + L.xhat);
    a.h = reinterpret_cast<bf16*>(ws + L.h);
    a.ev_h = reinterpret_cast<int32_t*>(ws + L.ev_h);
    a.ev_y = reinterpret_cast<int32_t*>(ws + L.ev_y);
    a.partial = reinterpret_cast<float*>(ws + L.partial);
    a.gu_part = reinterpret_cast<float*>(ws + L.gu_part);
    a.ev_gu = reinterpret_cast<int32_t*>(ws + L.ev_gu);
    a.gu_cap = L.gu_cap;
    a.mt_max = L.mt_max;
    a.num_ctas = st->sms;
    a.timeout_ns = timeout_ns_of(opts);
    a.fault_mode = opts ? opts->fault_mode : 0;
    a.fault_arg = opts ? opts->fault_arg : 0;
    a.trace = (opts && opts->trace && opts->trace_cap) ? static_cast<uint64_t*>(opts->trace) : nullptr;
    a.trace_cap = opts ? static_cast<int>(opts->trace_cap) : 0;
    CUtensorMap maps[7];
    if ((rc = make_map(&maps[0], w_gate, F, H, kTileM, "w_gate"))) return rc;
    if ((rc = make_map(&maps[1], w_up, F, H, kTileM, "w_up"))) return rc;
    if ((rc = make_map(&maps[2], w_down, H, F, kTileM, "w_down"))) return rc;
    if ((rc = make_map(&maps[3], a.xhat, B_max, H, kBBoxRows, "xhat"))) return rc;
    if ((rc = make_map(&maps[4], a.h, B_max, F, kBBoxRows, "h"))) return rc;
    a.b_wide = B_max >= kBBoxRowsWide ? 1 : 0;
    if (a.b_wide) {
        if ((rc = make_map(&maps[5], a.xhat, B_max, H, kBBoxRowsWide, "xhat"))) return rc;
        if ((rc = make_map(&maps[6], a.h, B_max, F, kBBoxRowsWide, "h"))) return rc;
    } else {
        maps[5] = maps[3];
        maps[6] = maps[4];
    }
    cudaError_t e = launch_mlp(a, maps, st->sms, smem, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e, "launch of the MLP chain kernel");
    return ET_OK;
}

int et_status(const void* workspace, void* stream, int32_t* code_out, int32_t* detail_out) {
    g_last_error.clear();
    if (!workspace || !code_out) return fail(ET_ERR_INVALID, "workspace and code_out must be non-NULL");
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e, "cudaStreamSynchronize");
    int32_t word[2] = {0, 0};
    e = cudaMemcpy(word, workspace, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail_cuda(e, "cudaMemcpy(status)");
    *code_out = word[0];
    if (detail_out) *detail_out = word[1];
    return ET_OK;
}

int et_reset_status(void* workspace, void* stream) {
    g_last_error.clear();
    if (!workspace) return fail(ET_ERR_INVALID, "workspace is NULL");
    cudaError_t e = cudaMemsetAsync(workspace, 0, 2 * sizeof(int32_t), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e, "cudaMemsetAsync(status)");
    return ET_OK;
}

}  // extern "C"

// ----------------------------------------------------------------------------
// Split-K GEMM without any allocation.
//
// Some callers cannot hand this library a workspace: a plugin or custom-op
// interface that passes only input and output buffers, or a code path that
// must not call cudaMalloc because allocating may synchronise the device or
// break a fixed memory plan.  For them, et_splitk_gemm_noalloc runs the same
// split-K kernel with its scratch (status word, tile counters, fp32 partial
// sums) in the file-scope device array below, which every GPU that loads the
// library keeps until the process exits.
// ----------------------------------------------------------------------------
static __device__ __align__(256) uint8_t g_splitk_noalloc_scratch[ET_SPLITK_NOALLOC_SCRATCH_BYTES];

namespace {

void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code the
// array's name is only a host-side stand-in, so the real address is looked up
// once per device, with that device current.  Like the library's other
// per-device state (kernel attributes), the address is kept for the life of
// the process: after cudaDeviceReset the process must be restarted.
int noalloc_scratch(int dev, void** out) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_noalloc_ptr[dev]) {
        void* ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_splitk_noalloc_scratch);
        if (e != cudaSuccess || ptr == nullptr)
            return fail_cuda(e, "cudaGetSymbolAddress(split-K scratch)");
        g_noalloc_ptr[dev] = ptr;
    }
    *out = g_noalloc_ptr[dev];
    return ET_OK;
}

}  // namespace

extern "C" int et_splitk_gemm_noalloc(const void* X, const void* Wt, void* Y, int M, int N, int K,
                                      int split, void* stream) {
    g_last_error.clear();
    if (!X || !Wt || !Y) return fail(ET_ERR_INVALID, "X, Wt and Y must be non-NULL");
    if (M < 0 || M > (1 << 20)) return fail(ET_ERR_INVALID, "M must be in [0, 2^20]");
    const size_t need = et_splitk_workspace_bytes(M > 0 ? M : 1, N, K, split);
    if (need == 0)
        return fail(ET_ERR_UNSUPPORTED,
                    "N must be a positive multiple of 128, split in [1, 16], K a multiple of 64*split");
    if (need > ET_SPLITK_NOALLOC_SCRATCH_BYTES)
        return fail(ET_ERR_WORKSPACE,
                    "et_splitk_gemm_noalloc: this shape needs " + std::to_string(need) +
                        " bytes of scratch but the built-in area holds " +
                        std::to_string(static_cast<size_t>(ET_SPLITK_NOALLOC_SCRATCH_BYTES)) +
                        " (use et_splitk_gemm with a workspace for larger shapes)");
    if (M == 0) return ET_OK;
    DeviceState* st = nullptr;
    int dev = 0;
    int rc = device_state(&st, &dev);
    if (rc) return rc;
    void* scratch = nullptr;
    if ((rc = noalloc_scratch(dev, &scratch))) return rc;
    // The array keeps the previous call's contents: zero the status word and
    // the tile counters (everything before the partial sums) for this call.
    const SplitKLayout L = splitk_layout(M, N, K, split);
    cudaError_t e = cudaMemsetAsync(scratch, 0, L.partial, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e, "cudaMemsetAsync(split-K scratch counters)");
    return et_splitk_gemm(X, Wt, Y, M, nullptr, M, N, K, split, scratch, need, nullptr, stream);
}

// The device status of the last et_splitk_gemm_noalloc call on the current
// device: synchronises `stream`, then reads the status word at the start of
// the built-in scratch array (cleared again by the next call).
extern "C" int et_splitk_noalloc_status(void* stream, int32_t* code_out, int32_t* detail_out) {
    g_last_error.clear();
    if (!code_out) return fail(ET_ERR_INVALID, "code_out must be non-NULL");
    DeviceState* st = nullptr;
    int dev = 0;
    int rc = device_state(&st, &dev);
    if (rc) return rc;
    void* scratch = nullptr;
    if ((rc = noalloc_scratch(dev, &scratch))) return rc;
    return et_status(scratch, stream, code_out, detail_out);
}
