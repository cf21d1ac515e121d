// rmsn_api.cu -- the C ABI: argument checks, the launch planner, the per-device property
// cache, the device error word and the exported entry points declared in include/rmsn.h.
//
// Checks run before anything is enqueued and return a status (the validation of
// FlashInfer PR #4480's wrapper: shape, dtype and alignment checked on the host, an
// unsupported hidden size rejected instead of launched).  The planner is a pure host
// function of (op, T, H, dtypes, SM count, shared memory per SM), testable without a GPU
// (Liger-Kernel PR #1336: fast-path eligibility helpers as pure functions).
#include <atomic>
#include <algorithm>
#include <mutex>
#include <vector>

#include "rmsn.h"
#include "rmsn_internal.h"
#include "rmsn_pipe.cuh"

// Device error word: bits set by kernels whose bounded waits ran out (rmsn_pipe.cuh).
__device__ unsigned int g_rmsn_error_word;

namespace {

using rmsn::Launch;

constexpr int64_t kDefaultSmemPerSm = 233472;   // 228 KiB on sm_100 / sm_103
constexpr int64_t kDefaultSmemPerCta = 232448;  // 227 KiB opt-in maximum per CTA
constexpr int64_t kSmemReservedPerCta = 1024;   // set aside by the driver for each CTA
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // every pipeline wait gives up after 1 s
constexpr int kWarpsPerSm = 16;  // the backward's consumer warps per SM (measured best on GB300)

// ------------------------------------------------------------------ policy defaults
struct Policy {
    int consumer_warps;  // 0: derived from H (target_nch vectors per lane)
    int ctas_per_sm;     // 0: derived (backward: kWarpsPerSm / consumer warps; forward: from
                         // the row size, about kFwdBytesInFlight of rows per SM)
    int max_stages;      // 0: derived (forward: two stages for rows of at most 4 KiB, else one)
    int target_nch;
    int max_nch;
};

// The forward's rows in flight per SM (ring stages of all its CTAs) for rows above 4 KiB:
// a launch-policy sweep on GB300 (bf16 and fp32, H 1024-8192, T 8192 and 65536) found the
// best CTAs per SM at about this many bytes of rows in flight, with one stage per CTA.
constexpr int64_t kFwdBytesInFlight = 48 << 10;
// The fused quant: stage bytes in flight per SM it aims for, and the warps per SM its
// register file holds at the kernel's bound of 72 registers per thread.
constexpr int64_t kFusedBytesInFlight = 64 << 10;
constexpr int64_t kFusedWarpsPerSm = 65536 / (72 * 32);

// Per op: FWD, BWD, FUSED, FWD_RESIDUAL, BWD_RESIDUAL.
constexpr int kOps = 5;
constexpr Policy kDefaultPolicy[kOps] = {
    {0, 0, 0, 6, 16},  // forward: at least 2 warps, about 6 vectors per lane, CTAs and
                       // stages from the row size
    {0, 0, 4, 2, 8},   // backward: 8 consumer warps at bf16 H 4096-6144, 16 per SM in all
    {0, 0, 0, 3, 8},   // fused quant: at most 3 vectors per lane (16 warps for the longest
                       // rows), stages and CTAs from the row size
    {0, 0, 2, 4, 16},  // residual forward: as the forward, two rows per stage
    {0, 0, 4, 2, 8},   // residual backward: as the backward (g_residual from global memory)
};
Policy g_policy[kOps] = {kDefaultPolicy[0], kDefaultPolicy[1], kDefaultPolicy[2],
                         kDefaultPolicy[3], kDefaultPolicy[4]};
std::mutex g_mu;

// Deterministic backward calls with T <= this take the one-launch column-task kernel
// (rmsn_set_small_t_max).
std::atomic<int64_t> g_small_t_max{256};  // measured break-even: T ~ 384-512 on GB300
bool small_t(int deterministic, int64_t T) {
    return deterministic && T <= g_small_t_max.load(std::memory_order_relaxed);
}

Policy policy(int op) {
    std::lock_guard<std::mutex> lk(g_mu);
    return g_policy[op];
}

// ------------------------------------------------------------------ device properties
struct DevProps {
    int sms = 0;
    int64_t smem_sm = 0;
    int64_t smem_cta = 0;
    unsigned* err = nullptr;
};
constexpr int kMaxDevices = 64;
DevProps g_props[kMaxDevices];
std::atomic<bool> g_props_ready[kMaxDevices];

const DevProps* props_of(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    if (g_props_ready[dev].load(std::memory_order_acquire)) return &g_props[dev];
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_props_ready[dev].load(std::memory_order_relaxed)) return &g_props[dev];
    DevProps p;
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
        cudaGetLastError();
        return nullptr;
    }
    p.sms = v;
    p.smem_sm = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) ==
                        cudaSuccess ? v : kDefaultSmemPerSm;
    p.smem_cta = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) ==
                         cudaSuccess ? v : kDefaultSmemPerCta;
    cudaGetLastError();
    g_props[dev] = p;
    g_props_ready[dev].store(true, std::memory_order_release);
    return &g_props[dev];
}

// The error word's device address for the current device (needs its context current).
unsigned* error_word(int dev) {
    static std::atomic<unsigned*> addr[kMaxDevices];
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    unsigned* p = addr[dev].load(std::memory_order_acquire);
    if (p) return p;
    void* a = nullptr;
    if (cudaGetSymbolAddress(&a, g_rmsn_error_word) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    addr[dev].store(static_cast<unsigned*>(a), std::memory_order_release);
    return static_cast<unsigned*>(a);
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
int esize(int dt) { return dt == RMSN_F32 ? 4 : 2; }
bool valid_dtype(int dt) { return dt == RMSN_F32 || dt == RMSN_BF16; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

template <size_t N>
int pick_nch(const int (&set)[N], int64_t need) {
    for (size_t i = 0; i < N; ++i)
        if (set[i] >= need) return set[i];
    return 0;
}

// The launch plan of one call.  Consumer warps: the smallest power of two (<= 8) whose
// lanes hold about `target_nch` 16-byte vectors of a row each (the backward: 16 for rows
// of at least 512 * target_nch vectors, and for some rows a count that is not a power of
// two, below); the chunk variant is the
// smallest compiled count that covers the row.  Shared memory per CTA: the ring header,
// the weight vector, and as many stages (<= max_stages) as the CTA's share of the SM
// holds (the backward at least two); fewer CTAs per SM if a share cannot hold two stages.
// The grid is clamped again at launch to what is resident at once (fit_grid).
int plan(int op, int64_t T, int64_t H, int x_dt, int w_dt, int sms, int64_t smem_sm,
         int64_t smem_cta, Launch* L, int64_t* ws_bytes) {
    if (op < 0 || op >= kOps) return RMSN_ERR_INVALID_ARG;
    if (!valid_dtype(x_dt) || !valid_dtype(w_dt)) return RMSN_ERR_INVALID_ARG;
    const bool is_bwd = op == RMSN_OP_BWD || op == RMSN_OP_BWD_RESIDUAL;
    if (op == RMSN_OP_FUSED_QUANT && (x_dt != RMSN_BF16 || w_dt != RMSN_BF16))
        return RMSN_ERR_INVALID_ARG;
    if (T < 0 || sms <= 0) return RMSN_ERR_INVALID_ARG;
    const int vec = 16 / esize(x_dt);
    if (H <= 0 || H > RMSN_MAX_H || H % vec != 0) return RMSN_ERR_UNSUPPORTED_SHAPE;
    if (is_bwd && x_dt == RMSN_F32 && H > 8192) return RMSN_ERR_UNSUPPORTED_SHAPE;
    if (op == RMSN_OP_FUSED_QUANT && H % 128 != 0) return RMSN_ERR_UNSUPPORTED_SHAPE;
    const Policy P = policy(op);
    const int64_t nvec = H / vec;
    int nw = P.consumer_warps;
    if (nw == 0) {
        nw = op == RMSN_OP_FWD ? 2 : 1;
        while (nw < 8 && cdiv(nvec, 32 * nw) > P.target_nch) nw *= 2;
        // backward rows that fill 16 warps at target_nch vectors per lane take 16 warps
        // (one CTA per SM), so every lane keeps its share of a row pair in registers
        if (is_bwd && nvec >= 16 * 32 * P.target_nch) nw = 16;
        // the fused quant: rows of more than 1024 vectors (bf16 H > 8192) take one CTA of 16
        // warps per SM (the 8-warp kernel would hold 4-8 vectors per lane and spill).
        // Measured on GB300 at T = 8192 / 32768: H 10240 159 -> 139 / 605 -> 526 us, H 12288
        // 162 -> 143 / 618 -> 549, H 16384 338 -> 193 / 1314 -> 739; H 8192 keeps 2 CTAs of 8
        if (op == RMSN_OP_FUSED_QUANT && nvec > 1024) nw = 16;
        // bf16 rows of about three vectors per lane at 8 warps (H 5632-6144) over a short
        // strip: one CTA of 16 warps per SM is faster up to T ~ 12288 (measured on GB300:
        // 14-16% at T = 2048, 8-9% at 4096, 2-4% at 8192, even at 16384, slower above), its
        // column reduce sums half as many chunks
        if (is_bwd && x_dt == RMSN_BF16 && nw == 8 && T <= 12288 &&
            cdiv(nvec, 32 * nw) == 3 && 4 * nvec >= 11 * 32 * (int64_t)nw)
            nw = 16;
        // backward rows that the power of two above spreads thinly: the fewest warps that
        // hold the row at target_nch vectors per lane, when those lanes are at least 7/8
        // full and 16 / nb CTAs of them give at least 14 warps per SM (bf16 H 1344-1536,
        // 2240-2560, 3136-3584; fp32 x at half those widths).  Where the power of two fills
        // more than 5/8 of its lanes, only over long strips (T >= 16384): more chunks cost
        // more than the fuller lanes save on short ones.  Measured on GB300, us per call:
        // H 2304 (5 warps, 3 CTAs) at T = 8192: 37.2 -> 32.0, at 65536: 212 -> 163; H 2560
        // at 4096: 25.9 -> 23.8, at 65536: 222 -> 167; H 1536 (3 warps, 5 CTAs) at 4096:
        // 20.6 -> 22.4, at 65536: 117 -> 113; H 3584 (7 warps, 2 CTAs) at 4096: 27.9 -> 28.7,
        // at 65536: 246 -> 229; H 3072 (6 warps, 12 per SM) was even, so it keeps 8.
        if (is_bwd && nw <= 8) {
            const int64_t nb = cdiv(nvec, 32 * P.target_nch);
            const int64_t lanes = 32 * (int64_t)nw * cdiv(nvec, 32 * nw);  // at the power of two
            if (nb < nw && 8 * nvec >= 7 * 32 * P.target_nch * nb &&
                nb * (kWarpsPerSm / nb) >= 14 && (8 * nvec <= 5 * lanes || T >= 16384))
                nw = (int)nb;
        }
        // short backward rows (1 or 2 warps) over short strips (fewer than 8 rows per chunk
        // at 16 / nw CTAs per SM): twice the warps in half the CTAs, so half as many chunk
        // partials to write and reduce.  Measured on GB300 (bf16, fp32 w): H 512 at T = 4096 /
        // 8192 / 16384 24.7 -> 16.6 / 25.8 -> 19.3 / 29.0 -> 25.1 us, H 256 at T = 8192 21.3 ->
        // 17.4, H 1024 at T = 4096 20.6 -> 18.0; at 13 or more rows per chunk the plan is best
        if (is_bwd && nw <= 2 && T < 8 * (int64_t)sms * (kWarpsPerSm / nw)) nw *= 2;
    }
    const int64_t need = cdiv(nvec, 32 * nw);
    int nch = 0;
    if (op == RMSN_OP_FWD || op == RMSN_OP_FWD_RESIDUAL) nch = pick_nch(rmsn::kFwdNch, need);
    else if (is_bwd) nch = pick_nch(rmsn::kBwdNch, need);
    else nch = pick_nch(rmsn::kFusedNch, need);
    if (nch == 0 || nch > P.max_nch) return RMSN_ERR_UNSUPPORTED_SHAPE;

    const int64_t row_bytes = H * esize(x_dt);
    const int64_t row_pad = cdiv(row_bytes, 128) * 128;
    // rows per stage: x; x and residual; x and dy (both backwards; the residual backward
    // reads g_residual from global memory)
    const int rows = op == RMSN_OP_FWD ? 1 : 2;
    const int64_t stage_bytes = rows * row_pad;
    const int64_t w_bytes = H * 4;  // w is staged in shared memory as FP32
    const int64_t data_off = rmsn::kRingHeader + cdiv(w_bytes, 128) * 128;
    // CTAs per SM: the policy's; or enough CTAs for kWarpsPerSm consumer warps per SM
    // (backward); or, for the forward, 8 for rows of at most 4 KiB and else about
    // kFwdBytesInFlight / row size (one stage each), fewer if shared memory or registers
    // run out (the grid is clamped to the resident CTAs at launch)
    const bool small_rows = row_bytes <= 4096;
    int cps = P.ctas_per_sm;
    // the residual forward (two rows per stage, two stages): 8 CTAs for rows of at most
    // 4 KiB, else 4.  Measured on GB300 at T = 8192 / 32768 against 4 CTAs: H 512 16.4 ->
    // 12.8 / 41.7 -> 28.7 us, H 1024 20.4 -> 16.5 / 59.4 -> 45.0, H 2048 even
    if (cps == 0 && op == RMSN_OP_FWD_RESIDUAL) cps = small_rows ? 8 : 4;
    if (cps == 0 && op == RMSN_OP_FWD)
        cps = small_rows ? 8
                         : (int)std::max<int64_t>(2, std::min<int64_t>(
                               8, (kFwdBytesInFlight + row_bytes / 2) / row_bytes));
    // the fused quant (one stage per CTA): about kFusedBytesInFlight of stages per SM, at
    // least two CTAs, at most as many as the registers hold.  Measured on GB300 at T = 8192
    // / 32768 against 3 CTAs of 2-8 warps at two vectors per lane: H 1024 34.2 -> 20.6 /
    // 110.8 -> 56.2 us (2 warps, 9 CTAs), H 2048 38.6 -> 30.3 / 129.0 -> 100.8 (4 warps,
    // 5 CTAs), H 3072 49.0 -> 41.1 / 169.4 -> 150.2 (4 warps, 5 CTAs), H 12288 246.6 ->
    // 162.3 / 951.5 -> 614.3 (2 CTAs, was 1); H 4096-8192 keep their plans (3 CTAs of 8
    // warps up to H 6144, 2 at H 8192, where 3 were 3-9% slower).
    if (cps == 0 && op == RMSN_OP_FUSED_QUANT && nw > 8) cps = 1;  // 16 warps: one CTA
    if (cps == 0 && op == RMSN_OP_FUSED_QUANT) {
        const int64_t by_bytes = (kFusedBytesInFlight + stage_bytes / 2) / stage_bytes;
        const int64_t by_regs = kFusedWarpsPerSm / (nw + 1);  // + the producer warp
        cps = (int)std::max<int64_t>(2, std::min(by_bytes, by_regs));
    }
    if (cps == 0) cps = nw >= kWarpsPerSm ? 1 : kWarpsPerSm / nw;
    // the fused quant's 16-warp CTA: two stages while they stay within about 96 KiB (H up
    // to 12288: 143 against 155 us at T = 8192), else one (H 16384: 193 against 199)
    const int max_stages =
        P.max_stages > 0 ? P.max_stages
        : (op == RMSN_OP_FUSED_QUANT) ? (nw > 8 && stage_bytes <= (96 << 10) / 2 ? 2 : 1)
        : (small_rows ? 2 : 1);
    auto stages_for = [&](int c) -> int64_t {
        int64_t share = smem_sm / c - kSmemReservedPerCta;
        if (share > smem_cta) share = smem_cta;
        return (share - data_off) / stage_bytes;
    };
    // the backward holds two rows' stages at once (it takes rows two at a time)
    const int64_t min_stages = is_bwd ? 2 : 1;
    // room for two stages per CTA (the forward and the fused quant: for as many as they
    // will use)
    const int64_t want_stages = (op == RMSN_OP_FWD || op == RMSN_OP_FUSED_QUANT)
                                    ? std::max<int64_t>(1, std::min<int64_t>(2, max_stages))
                                    : 2;
    while (cps > 1 && stages_for(cps) < want_stages) --cps;
    int64_t stages = stages_for(cps);
    if (stages < min_stages) return RMSN_ERR_UNSUPPORTED_SHAPE;
    if (stages > max_stages) stages = max_stages > min_stages ? max_stages : min_stages;

    int64_t grid = (int64_t)sms * cps;
    if (grid > T) grid = T;
    if (grid < 1) grid = 1;
    L->nw = nw;
    L->nch = nch;
    // the backward takes bf16 rows of three vectors per lane one at a time with 16 warps, and
    // with fewer when the lanes' third vectors are at least 3/4 full (measured on GB300: with
    // 8 warps at 2.5 vectors per lane (H = 5120) pairs are 15% faster, at 3 (H = 6144) single
    // rows 3-9% faster; with 16 warps single rows are 4-10% faster at H 8704-10240)
    L->single = is_bwd && x_dt == RMSN_BF16 && nch == 3 &&
                (nw == 16 || 4 * nvec >= 11 * 32 * (int64_t)nw);
    L->stages = (int)stages;
    L->ctas_per_sm = cps;
    L->sms = sms;
    L->row_bytes = (uint32_t)row_bytes;
    L->stage_bytes = (uint32_t)stage_bytes;
    L->w_bytes = (uint32_t)w_bytes;
    L->data_off = (uint32_t)data_off;
    L->grid = grid;
    L->smem = data_off + stages * stage_bytes;
    L->err = nullptr;
    L->limit_ns = kWaitLimitNs;
    // the backward's workspace: the chunks' (high, low) partial rows
    if (ws_bytes) *ws_bytes = is_bwd ? grid * H * 4 * 2 : 0;
    return RMSN_OK;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? RMSN_OK : RMSN_ERR_CUDA; }

// Plans a call on the current device and fills in the device-dependent fields.
int plan_current(int op, int64_t T, int64_t H, int x_dt, int w_dt, Launch* L, int64_t* ws) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return RMSN_ERR_CUDA;
    }
    const DevProps* p = props_of(dev);
    if (!p) return RMSN_ERR_CUDA;
    int st = plan(op, T, H, x_dt, w_dt, p->sms, p->smem_sm, p->smem_cta, L, ws);
    if (st != RMSN_OK) return st;
    L->err = error_word(dev);
    return L->err ? RMSN_OK : RMSN_ERR_CUDA;
}

}  // namespace

namespace rmsn {

// Self-test of the bounded wait: one thread waits on an mbarrier that expects an arrival
// nobody makes (no copy is in flight), gives up after `limit_ns`, and reports it through
// the error word exactly as a pipeline wait does.
__global__ void rmsn_wait_selftest_kernel(unsigned* err, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    if (!mbar_wait(&bar, 0u, limit_ns)) atomicOr(err, ERR_WAIT_FULL);
}

cudaError_t launch_wait_selftest(unsigned* err, uint64_t limit_ns, cudaStream_t s) {
    rmsn_wait_selftest_kernel<<<1, 32, 0, s>>>(err, limit_ns);
    return cudaGetLastError();
}

cudaError_t fit_grid(const void* kernel, const Launch& L, int threads, int64_t* grid) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const DevProps* p = props_of(dev);
    if (!p) return cudaErrorInvalidDevice;
    // The dynamic shared memory limit is a per-kernel attribute: it is raised once to the
    // device's opt-in maximum (a limit, not a reservation), never lowered, so any plan's
    // size launches.  Occupancy is cached per (kernel, threads, shared memory).
    struct Occ {
        int dev;
        const void* k;
        int threads;
        int64_t smem;
        int occ;
    };
    struct Opted {
        int dev;
        const void* k;
    };
    static std::vector<Occ> occs;
    static std::vector<Opted> opted;
    static std::mutex mu;
    std::lock_guard<std::mutex> lk(mu);
    int occ = 0;
    for (const auto& x : occs)
        if (x.dev == dev && x.k == kernel && x.threads == threads && x.smem == L.smem) {
            occ = x.occ;
            break;
        }
    if (occ == 0) {
        bool done = false;
        for (const auto& x : opted)
            if (x.dev == dev && x.k == kernel) done = true;
        if (!done) {
            // the opt-in maximum covers static and dynamic shared memory together
            cudaFuncAttributes fa{};
            e = cudaFuncGetAttributes(&fa, kernel);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)(p->smem_cta - (int64_t)fa.sharedSizeBytes));
            if (e != cudaSuccess) return e;
            opted.push_back({dev, kernel});
        }
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, threads, (size_t)L.smem);
        if (e != cudaSuccess) return e;
        if (occ < 1) return cudaErrorInvalidConfiguration;
        occs.push_back({dev, kernel, threads, L.smem, occ});
    }
    const int64_t resident = (int64_t)L.sms * occ;
    *grid = L.grid < resident ? L.grid : resident;
    return cudaSuccess;
}

}  // namespace rmsn

extern "C" {

const char* rmsn_status_string(int status) {
    switch (status) {
        case RMSN_OK: return "ok";
        case RMSN_ERR_INVALID_ARG: return "invalid argument (null pointer, dtype, T, ld or eps)";
        case RMSN_ERR_UNSUPPORTED_SHAPE:
            return "unsupported shape (H must be a positive multiple of the 16-byte vector, "
                   "at most 16384; the fused quant needs H % 128 == 0; the fp32 backward "
                   "at most 8192)";
        case RMSN_ERR_MISALIGNED: return "misaligned pointer (16-byte alignment required)";
        case RMSN_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than rmsnorm_bwd_workspace_bytes";
        case RMSN_ERR_CUDA: return "CUDA error (launch or runtime call failed)";
        case RMSN_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait ran out (device error word set)";
        case RMSN_ERR_SCRATCH_LIMIT:
            return "rmsnorm_bwd_noalloc: this T and H need more scratch than its fixed 16 MiB "
                   "(use rmsnorm_bwd with a caller workspace)";
        default: return "unknown status";
    }
}

int rmsn_plan(int op, int64_t T, int64_t H, int x_dtype, int w_dtype, int compensated,
              int sm_count, rmsn_plan_t* out) {
    (void)compensated;
    if (!out) return RMSN_ERR_INVALID_ARG;
    Launch L{};
    int64_t ws = 0;
    int st = plan(op, T, H, x_dtype, w_dtype, sm_count, kDefaultSmemPerSm, kDefaultSmemPerCta,
                  &L, &ws);
    if (st != RMSN_OK) return st;
    out->vec_elems = 16 / esize(x_dtype);
    out->consumer_warps = L.nw;
    out->chunks_per_lane = L.nch;
    const bool is_bwd = op == RMSN_OP_BWD || op == RMSN_OP_BWD_RESIDUAL;
    out->threads = is_bwd ? L.nw * 32 : L.nw * 32 + 32;  // backward: no producer warp
    out->stages = L.stages;
    out->ctas_per_sm = L.ctas_per_sm;
    out->grid = L.grid;
    out->smem_bytes = L.smem;
    out->workspace_bytes = ws;
    return RMSN_OK;
}

int rmsn_set_policy(int op, int consumer_warps, int ctas_per_sm, int max_stages) {
    if (op < 0 || op >= kOps) return RMSN_ERR_INVALID_ARG;
    const bool is_bwd = op == RMSN_OP_BWD || op == RMSN_OP_BWD_RESIDUAL;
    // the backward takes any number of consumer warps up to 16, the fused quant 1, 2, 4, 8
    // or 16 (16 for rows of 1024-2048 vectors), the forwards 1, 2, 4, 8
    const int max_warps = (is_bwd || op == RMSN_OP_FUSED_QUANT) ? 16 : 8;
    if (consumer_warps < 0 || consumer_warps > max_warps ||
        (!is_bwd && (consumer_warps & (consumer_warps - 1)) != 0))
        return RMSN_ERR_INVALID_ARG;
    if (ctas_per_sm < 0 || ctas_per_sm > 16 || max_stages < 0 || max_stages > 32)
        return RMSN_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_mu);
    Policy p = kDefaultPolicy[op];
    p.consumer_warps = consumer_warps;
    if (ctas_per_sm) p.ctas_per_sm = ctas_per_sm;
    if (max_stages) p.max_stages = max_stages;
    g_policy[op] = p;
    return RMSN_OK;
}

int rmsn_set_small_t_max(int64_t t_max) {
    if (t_max < 0 || t_max > (1 << 20)) return RMSN_ERR_INVALID_ARG;
    g_small_t_max.store(t_max, std::memory_order_relaxed);
    return RMSN_OK;
}

int64_t rmsn_small_t_max(void) { return g_small_t_max.load(std::memory_order_relaxed); }

int rmsn_selftest_wait_timeout(uint64_t limit_ns, rmsn_stream_t stream) {
    if (limit_ns == 0 || limit_ns > kWaitLimitNs) return RMSN_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return RMSN_ERR_CUDA;
    }
    unsigned* w = error_word(dev);
    if (!w) return RMSN_ERR_CUDA;
    return from_cuda(rmsn::launch_wait_selftest(w, limit_ns, reinterpret_cast<cudaStream_t>(stream)));
}

int rmsn_device_status(rmsn_stream_t stream, unsigned* flags) {
    if (!flags) return RMSN_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return RMSN_ERR_CUDA;
    }
    unsigned* w = error_word(dev);
    if (!w) return RMSN_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned v = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess ||
        cudaMemcpy(&v, w, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(w, 0, sizeof v) != cudaSuccess) {
        cudaGetLastError();
        return RMSN_ERR_CUDA;
    }
    *flags = v;
    return v ? RMSN_ERR_DEVICE_TIMEOUT : RMSN_OK;
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
    Launch L{};
    int st = plan_current(RMSN_OP_FWD, T, H, x_dtype, w_dtype, &L, nullptr);
    if (st != RMSN_OK) return st;
    return from_cuda(rmsn::launch_fwd(L, x, x_dtype, w, w_dtype, y, rstd, T, H, eps,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

size_t rmsnorm_bwd_workspace_bytes(int64_t T, int64_t H, int compensated, int device) {
    (void)compensated;
    if (T <= 0 || H <= 0 || H > RMSN_MAX_H || H % 4 != 0) return 0;
    const DevProps* p = props_of(device);
    if (!p) return 0;
    // The largest workspace any plan of rmsnorm_bwd or rmsnorm_bwd_residual needs for this
    // (T, H) over the dtype pairs; each grows with T (min(T, SMs x CTAs per SM) chunks), so
    // this bounds every call with T' <= T.
    int64_t best = 0;
    for (int op : {(int)RMSN_OP_BWD, (int)RMSN_OP_BWD_RESIDUAL})
        for (int xd : {(int)RMSN_F32, (int)RMSN_BF16})
            for (int wd : {(int)RMSN_F32, (int)RMSN_BF16}) {
                Launch L{};
                int64_t ws = 0;
                if (plan(op, T, H, xd, wd, p->sms, p->smem_sm, p->smem_cta, &L, &ws) == RMSN_OK)
                    best = std::max(best, ws);
            }
    return (size_t)best;
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
    if (!workspace) return workspace_bytes ? RMSN_ERR_INVALID_ARG : RMSN_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned(workspace, 16)) return RMSN_ERR_MISALIGNED;
    Launch L{};
    int64_t need = 0;
    int st = plan_current(RMSN_OP_BWD, T, H, x_dtype, w_dtype, &L, &need);
    if (st != RMSN_OK) return st;
    if ((int64_t)workspace_bytes < need) return RMSN_ERR_WORKSPACE_TOO_SMALL;
    if (small_t(deterministic, T))
        return from_cuda(rmsn::launch_bwd_small(dy, x, x_dtype, w, w_dtype, rstd, dx, dw, T, H,
                                                compensated, s));
    return from_cuda(rmsn::launch_bwd(L, dy, x, x_dtype, w, w_dtype, rstd, dx, dw, T, H,
                                      deterministic, compensated,
                                      static_cast<float*>(workspace), s));
}

int rmsnorm_fwd_residual(const void* x, const void* residual, int x_dtype, const void* w,
                         int w_dtype, void* y, void* h_new, float* rstd, int64_t T, int64_t H,
                         float eps, rmsn_stream_t stream) {
    if (!valid_dtype(x_dtype) || !valid_dtype(w_dtype)) return RMSN_ERR_INVALID_ARG;
    if (T < 0 || !(eps >= 0.f) || eps == __builtin_huge_valf()) return RMSN_ERR_INVALID_ARG;
    if (H <= 0 || H > RMSN_MAX_H || H % (16 / esize(x_dtype)) != 0) return RMSN_ERR_UNSUPPORTED_SHAPE;
    if (T == 0) return RMSN_OK;
    if (!x || !residual || !w || !y || !h_new || !rstd) return RMSN_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(residual, 16) || !aligned(w, 16) || !aligned(y, 16) ||
        !aligned(h_new, 16) || !aligned(rstd, 4))
        return RMSN_ERR_MISALIGNED;
    Launch L{};
    int st = plan_current(RMSN_OP_FWD_RESIDUAL, T, H, x_dtype, w_dtype, &L, nullptr);
    if (st != RMSN_OK) return st;
    return from_cuda(rmsn::launch_fwd(L, x, x_dtype, w, w_dtype, y, rstd, T, H, eps,
                                      reinterpret_cast<cudaStream_t>(stream), residual, h_new));
}

int rmsnorm_bwd_residual(const void* dy, const void* h, int x_dtype, const void* w, int w_dtype,
                         const float* rstd, const void* g_residual, void* dx_total, float* dw,
                         int64_t T, int64_t H, int deterministic, int compensated,
                         void* workspace, size_t workspace_bytes, rmsn_stream_t stream) {
    if (!valid_dtype(x_dtype) || !valid_dtype(w_dtype) || T < 0) return RMSN_ERR_INVALID_ARG;
    if (H <= 0 || H > RMSN_MAX_H || H % (16 / esize(x_dtype)) != 0) return RMSN_ERR_UNSUPPORTED_SHAPE;
    if (!dw) return RMSN_ERR_INVALID_ARG;
    if (!aligned(dw, 16)) return RMSN_ERR_MISALIGNED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (T == 0) return from_cuda(cudaMemsetAsync(dw, 0, (size_t)H * sizeof(float), s));
    if (!dy || !h || !w || !rstd || !g_residual || !dx_total) return RMSN_ERR_INVALID_ARG;
    if (!aligned(dy, 16) || !aligned(h, 16) || !aligned(w, 16) || !aligned(g_residual, 16) ||
        !aligned(dx_total, 16) || !aligned(rstd, 4))
        return RMSN_ERR_MISALIGNED;
    if (!workspace) return workspace_bytes ? RMSN_ERR_INVALID_ARG : RMSN_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned(workspace, 16)) return RMSN_ERR_MISALIGNED;
    Launch L{};
    int64_t need = 0;
    int st = plan_current(RMSN_OP_BWD_RESIDUAL, T, H, x_dtype, w_dtype, &L, &need);
    if (st != RMSN_OK) return st;
    if ((int64_t)workspace_bytes < need) return RMSN_ERR_WORKSPACE_TOO_SMALL;
    if (small_t(deterministic, T))
        return from_cuda(rmsn::launch_bwd_small(dy, h, x_dtype, w, w_dtype, rstd, dx_total, dw, T,
                                                H, compensated, s, g_residual));
    return from_cuda(rmsn::launch_bwd(L, dy, h, x_dtype, w, w_dtype, rstd, dx_total, dw, T, H,
                                      deterministic, compensated,
                                      static_cast<float*>(workspace), s, g_residual));
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
    Launch L{};
    int st = plan_current(RMSN_OP_FUSED_QUANT, T, H, RMSN_BF16, RMSN_BF16, &L, nullptr);
    if (st != RMSN_OK) return st;
    return from_cuda(rmsn::launch_fused(L, x, residual, w, q, block_scale, scale_ld, normed, T, H,
                                        eps, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

// ---------------------------------------------------------- allocation-free backward
// Scratch of rmsnorm_bwd_noalloc, for callers that cannot allocate a workspace (see
// include/rmsn.h).  It lives in device memory reserved when the library is loaded; the
// name is a host-side stand-in, so the device address is looked up per device below and
// only that address is handed to the kernels.
static __device__ __align__(256) unsigned char g_bwd_noalloc_scratch[RMSN_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of the scratch array on `dev` (which must be current); looked up once per
// device.  nullptr if the lookup fails.
void* noalloc_scratch(int dev) {
    static std::atomic<void*> addr[kMaxDevices];
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    void* p = addr[dev].load(std::memory_order_acquire);
    if (p) return p;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_bwd_noalloc_scratch) != cudaSuccess || !ptr) {
        cudaGetLastError();
        return nullptr;
    }
    addr[dev].store(ptr, std::memory_order_release);
    return ptr;
}

}  // namespace

extern "C" int rmsnorm_bwd_noalloc(const void* dy, const void* x, int x_dtype, const void* w,
                                   int w_dtype, const float* rstd, void* dx, float* dw, int64_t T,
                                   int64_t H, int compensated, rmsn_stream_t stream) {
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
    Launch L{};
    int64_t need = 0;
    int st = plan_current(RMSN_OP_BWD, T, H, x_dtype, w_dtype, &L, &need);
    if (st != RMSN_OK) return st;
    // The address lookup comes first on every route, so a device's first call always does
    // it (the header asks for that first call to precede any stream capture).
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return RMSN_ERR_CUDA;
    }
    void* scratch = noalloc_scratch(dev);
    if (!scratch) return RMSN_ERR_CUDA;
    // The one-launch small-T kernel needs no scratch, so the limit applies to the strip route
    // only.
    if (small_t(1, T))
        return from_cuda(rmsn::launch_bwd_small(dy, x, x_dtype, w, w_dtype, rstd, dx, dw, T, H,
                                                compensated, s));
    if (need > (int64_t)RMSN_NOALLOC_SCRATCH_BYTES) return RMSN_ERR_SCRATCH_LIMIT;
    return from_cuda(rmsn::launch_bwd(L, dy, x, x_dtype, w, w_dtype, rstd, dx, dw, T, H,
                                      /*deterministic=*/1, compensated,
                                      static_cast<float*>(scratch), s));
}
