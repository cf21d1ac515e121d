// rmsn_api.cu -- the C ABI: argument checks, the launch planner, the per-device SM-count
// cache and the exported entry points declared in include/rmsn.h.
//
// Checks run before anything is enqueued and return a status (the validation of
// FlashInfer PR #4480's wrapper: shape, dtype and alignment checked on the host, an
// unsupported hidden size rejected instead of launched).  The planner is a pure host
// function of (op, T, H, dtypes, flags, SM count), testable without a GPU
// (Liger-Kernel PR #1336: fast-path eligibility helpers as pure functions).
#include <atomic>
#include <mutex>

#include "rmsn.h"
#include "rmsn_internal.h"

namespace {

using rmsn::Launch;

// ------------------------------------------------------------------ policy defaults
struct Policy {
    int threads;
    int ctas_per_sm;
    int wpr;        // 0: smallest count that fits the per-lane chunk budget
    int max_nch;    // per-lane chunk budget (registers)
};

// Defaults per op: FWD, BWD, FUSED.  Threads and CTAs per SM size the persistent grid;
// the chunk budget bounds the per-lane register row cache.
constexpr Policy kDefaultPolicy[3] = {
    {256, 4, 0, 8},  // forward: row cache of up to 8 x 16 B per lane
    {256, 2, 0, 4},  // backward: x and dy caches plus the dw accumulators
    {256, 4, 0, 8},  // fused: x and residual caches
};
Policy g_policy[3] = {kDefaultPolicy[0], kDefaultPolicy[1], kDefaultPolicy[2]};
std::mutex g_policy_mu;

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

int sm_count_of(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return 0;
    int v = g_sm_count[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 0;
    }
    g_sm_count[dev].store(n, std::memory_order_relaxed);
    return n;
}

int current_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return sm_count_of(dev);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int esize(int dt) { return dt == RMSN_F32 ? 4 : 2; }

bool valid_dtype(int dt) { return dt == RMSN_F32 || dt == RMSN_BF16; }

template <size_t N>
int pick_nch(const int (&set)[N], int need) {
    for (size_t i = 0; i < N; ++i)
        if (set[i] >= need) return set[i];
    return 0;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Chooses warps per row and the chunk variant: the smallest power-of-two warp count whose
// per-lane chunk count fits the budget (so a row is read by as few lanes as possible, each
// with a long run of 16-byte loads).
int plan_geometry(int op, int64_t H, int vec, const Policy& P, Launch* L) {
    const int64_t nvec = H / vec;
    const int max_nch = P.max_nch;
    int wpr = P.wpr;
    if (wpr == 0) {
        for (wpr = 1; wpr <= 16; wpr *= 2)
            if (cdiv(nvec, 32 * wpr) <= max_nch) break;
        if (wpr > 16) wpr = 16;  // over budget: the widest group, the largest compiled variant
    }
    const int need = (int)cdiv(nvec, 32 * wpr);
    int nch = 0;
    if (op == RMSN_OP_FWD) nch = pick_nch(rmsn::kFwdNch, need);
    else if (op == RMSN_OP_BWD) nch = pick_nch(rmsn::kBwdNch, need);
    else nch = pick_nch(rmsn::kFusedNch, need);
    if (nch == 0) return RMSN_ERR_UNSUPPORTED_SHAPE;
    int threads = P.threads < 32 * wpr ? 32 * wpr : P.threads;
    if (threads % (32 * wpr) != 0 || threads > 512) return RMSN_ERR_UNSUPPORTED_SHAPE;
    const int groups = threads / (32 * wpr);
    if (wpr > 1 && groups > 15) return RMSN_ERR_UNSUPPORTED_SHAPE;  // named barriers 1..15
    L->wpr = wpr;
    L->nch = nch;
    L->threads = threads;
    L->groups = groups;
    return RMSN_OK;
}

int plan(int op, int64_t T, int64_t H, int x_dt, int w_dt, int comp, int sms, Launch* L,
         int64_t* ws_bytes) {
    if (op < 0 || op > 2) return RMSN_ERR_INVALID_ARG;
    if (!valid_dtype(x_dt) || !valid_dtype(w_dt)) return RMSN_ERR_INVALID_ARG;
    if (op == RMSN_OP_FUSED_QUANT && (x_dt != RMSN_BF16 || w_dt != RMSN_BF16))
        return RMSN_ERR_INVALID_ARG;
    if (T < 0 || sms <= 0) return RMSN_ERR_INVALID_ARG;
    const int vec = 16 / esize(x_dt);
    if (H <= 0 || H > RMSN_MAX_H || H % vec != 0) return RMSN_ERR_UNSUPPORTED_SHAPE;
    if (op == RMSN_OP_FUSED_QUANT && H % 128 != 0) return RMSN_ERR_UNSUPPORTED_SHAPE;
    Policy P;
    {
        std::lock_guard<std::mutex> lk(g_policy_mu);
        P = g_policy[op];
    }
    int st = plan_geometry(op, H, vec, P, L);
    if (st != RMSN_OK) return st;
    const int64_t cap = (int64_t)sms * P.ctas_per_sm;
    int64_t grid = cdiv(T, L->groups);
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    L->grid = grid;
    L->smem = 0;
    if (ws_bytes) *ws_bytes = 0;
    if (op == RMSN_OP_BWD) {
        const int64_t parts = comp ? 2 : 1;
        if (L->groups > 1) L->smem = H * 4 * parts;  // group fold buffer
        if (ws_bytes) *ws_bytes = grid * H * 4 * parts;
    }
    return RMSN_OK;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? RMSN_OK : RMSN_ERR_CUDA; }

}  // namespace

extern "C" {

const char* rmsn_status_string(int status) {
    switch (status) {
        case RMSN_OK: return "ok";
        case RMSN_ERR_INVALID_ARG: return "invalid argument (null pointer, dtype, T or eps)";
        case RMSN_ERR_UNSUPPORTED_SHAPE:
            return "unsupported shape (H must be a positive multiple of the 16-byte vector, "
                   "at most 16384; the fused quant needs H % 128 == 0)";
        case RMSN_ERR_MISALIGNED: return "misaligned pointer (16-byte alignment required)";
        case RMSN_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than rmsnorm_bwd_workspace_bytes";
        case RMSN_ERR_CUDA: return "CUDA error (launch or runtime call failed)";
        default: return "unknown status";
    }
}

int rmsn_plan(int op, int64_t T, int64_t H, int x_dtype, int w_dtype, int compensated,
              int sm_count, rmsn_plan_t* out) {
    if (!out) return RMSN_ERR_INVALID_ARG;
    Launch L{};
    int64_t ws = 0;
    int st = plan(op, T, H, x_dtype, w_dtype, compensated, sm_count, &L, &ws);
    if (st != RMSN_OK) return st;
    Policy P;
    {
        std::lock_guard<std::mutex> lk(g_policy_mu);
        P = g_policy[op];
    }
    out->vec_elems = 16 / esize(x_dtype);
    out->warps_per_row = L.wpr;
    out->chunks_per_lane = L.nch;
    out->threads = L.threads;
    out->rows_per_cta = L.groups;
    out->ctas_per_sm = P.ctas_per_sm;
    out->grid = L.grid;
    out->smem_bytes = L.smem;
    out->workspace_bytes = ws;
    return RMSN_OK;
}

int rmsn_set_policy(int op, int threads, int ctas_per_sm, int warps_per_row) {
    if (op < 0 || op > 2) return RMSN_ERR_INVALID_ARG;
    if (threads < 0 || threads > 512 || threads % 32 != 0) return RMSN_ERR_INVALID_ARG;
    if (ctas_per_sm < 0 || ctas_per_sm > 32) return RMSN_ERR_INVALID_ARG;
    if (warps_per_row < 0 || warps_per_row > 16 || (warps_per_row & (warps_per_row - 1)) != 0)
        return RMSN_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_policy_mu);
    Policy p = kDefaultPolicy[op];
    if (threads) p.threads = threads;
    if (ctas_per_sm) p.ctas_per_sm = ctas_per_sm;
    p.wpr = warps_per_row;
    g_policy[op] = p;
    return RMSN_OK;
}

int rmsnorm_fwd(const void* x, int x_dtype, const void* w, int w_dtype, void* y, float* rstd,
                int64_t T, int64_t H, float eps, rmsn_stream_t stream) {
    if (!valid_dtype(x_dtype) || !valid_dtype(w_dtype)) return RMSN_ERR_INVALID_ARG;
    if (T < 0 || !(eps >= 0.f) || eps == __builtin_huge_valf()) return RMSN_ERR_INVALID_ARG;
    if (H <= 0 || H > RMSN_MAX_H || H % (16 / esize(x_dtype)) != 0) return RMSN_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return RMSN_OK;
    if (!x || !w || !y || !rstd) return RMSN_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 16) || !aligned(rstd, 4))
        return RMSN_ERR_MISALIGNED;
    const int sms = current_sm_count();
    if (sms <= 0) return RMSN_ERR_CUDA;
    Launch L{};
    int st = plan(RMSN_OP_FWD, T, H, x_dtype, w_dtype, 0, sms, &L, nullptr);
    if (st != RMSN_OK) return st;
    return from_cuda(rmsn::launch_fwd(L, x, x_dtype, w, w_dtype, y, rstd, T, H, eps,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

size_t rmsnorm_bwd_workspace_bytes(int64_t T, int64_t H, int compensated, int device) {
    if (T <= 0 || H <= 0 || H > RMSN_MAX_H || H % 4 != 0) return 0;
    const int sms = sm_count_of(device);
    if (sms <= 0) return 0;
    Policy P;
    {
        std::lock_guard<std::mutex> lk(g_policy_mu);
        P = g_policy[RMSN_OP_BWD];
    }
    // The chunk count never exceeds min(T, SMs * CTAs per SM) whatever the dtypes, and
    // grows with T, so this bounds every call with T' <= T.
    int64_t chunks = (int64_t)sms * P.ctas_per_sm;
    if (chunks > T) chunks = T;
    return (size_t)(chunks * H * 4 * (compensated ? 2 : 1));
}

int rmsnorm_bwd(const void* dy, const void* x, int x_dtype, const void* w, int w_dtype,
                const float* rstd, void* dx, float* dw, int64_t T, int64_t H, int deterministic,
                int compensated, void* workspace, size_t workspace_bytes, rmsn_stream_t stream) {
    if (!valid_dtype(x_dtype) || !valid_dtype(w_dtype) || T < 0) return RMSN_ERR_INVALID_ARG;
    if (H <= 0 || H > RMSN_MAX_H || H % (16 / esize(x_dtype)) != 0) return RMSN_ERR_UNSUPPORTED_SHAPE;
    if (!dw) return RMSN_ERR_INVALID_ARG;
    if (!aligned(dw, 16)) return RMSN_ERR_MISALIGNED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (T == 0) return from_cuda(cudaMemsetAsync(dw, 0, (size_t)H * sizeof(float), s));
    if (!dy || !x || !w || !rstd || !dx) return RMSN_ERR_INVALID_ARG;
    if (!aligned(dy, 16) || !aligned(x, 16) || !aligned(w, 16) || !aligned(dx, 16) ||
        !aligned(rstd, 4))
        return RMSN_ERR_MISALIGNED;
    const int sms = current_sm_count();
    if (sms <= 0) return RMSN_ERR_CUDA;
    Launch L{};
    int64_t need = 0;
    int st = plan(RMSN_OP_BWD, T, H, x_dtype, w_dtype, compensated, sms, &L, &need);
    if (st != RMSN_OK) return st;
    if (deterministic) {
        if (!workspace) return workspace_bytes ? RMSN_ERR_INVALID_ARG : RMSN_ERR_WORKSPACE_TOO_SMALL;
        if (!aligned(workspace, 16)) return RMSN_ERR_MISALIGNED;
        if ((int64_t)workspace_bytes < need) return RMSN_ERR_WORKSPACE_TOO_SMALL;
    }
    return from_cuda(rmsn::launch_bwd(L, dy, x, x_dtype, w, w_dtype, rstd, dx, dw, T, H,
                                      deterministic, compensated,
                                      static_cast<float*>(workspace), s));
}

int fused_add_rmsnorm_fp8_block_quant(const void* x, void* residual, const void* w, uint8_t* q,
                                      float* block_scale, int64_t scale_ld, void* normed,
                                      int64_t T, int64_t H, float eps, rmsn_stream_t stream) {
    if (T < 0 || !(eps >= 0.f) || eps == __builtin_huge_valf()) return RMSN_ERR_INVALID_ARG;
    if (H <= 0 || H > RMSN_MAX_H || H % 128 != 0) return RMSN_ERR_UNSUPPORTED_SHAPE;
    if (scale_ld < (T + 3) / 4 * 4) return RMSN_ERR_INVALID_ARG;
    if (T == 0) return RMSN_OK;
    if (!x || !residual || !w || !q || !block_scale || !normed) return RMSN_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(residual, 16) || !aligned(w, 16) || !aligned(normed, 16) ||
        !aligned(q, 16) || !aligned(block_scale, 4))
        return RMSN_ERR_MISALIGNED;
    const int sms = current_sm_count();
    if (sms <= 0) return RMSN_ERR_CUDA;
    Launch L{};
    int st = plan(RMSN_OP_FUSED_QUANT, T, H, RMSN_BF16, RMSN_BF16, 0, sms, &L, nullptr);
    if (st != RMSN_OK) return st;
    return from_cuda(rmsn::launch_fused(L, x, residual, w, q, block_scale, scale_ld, normed, T, H,
                                        eps, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
