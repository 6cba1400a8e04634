// C ABI of the KDA library: argument validation and dispatch to the kernels.
//
// Everything here runs on the host, allocates nothing and never synchronises.
// Argument errors return before any CUDA call is made.
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "kda_internal.cuh"

using kda::segment_shape;
#include <nvtx3/nvToolsExt.h>

namespace {

thread_local char g_last_error[256] = "";

void set_last_error(const char* msg) {
    strncpy(g_last_error, msg, sizeof(g_last_error) - 1);
    g_last_error[sizeof(g_last_error) - 1] = '\0';
}

// An NVTX range around each entry point (named after it), so a timeline
// profiler shows every library call; free when no tool is attached.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// [p, p + n) and [q, q + m) overlap (both non-empty)?
bool overlaps(const void* p, size_t n, const void* q, size_t m) {
    if (!p || !q || n == 0 || m == 0) return false;
    uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
    return a < b + m && b < a + n;
}

// n = a * b * c * d with overflow detection (all factors >= 0).
bool mul_ok(size_t* out, size_t a, size_t b, size_t c = 1, size_t d = 1) {
    const size_t lim = (size_t)1 << 62;
    size_t r = a;
    for (size_t f : {b, c, d}) {
        if (f != 0 && r > lim / f) return false;
        r *= f;
    }
    *out = r;
    return true;
}

kda_status_t fail(kda_status_t s, const char* why) {
    set_last_error(why);
    return s;
}

kda_status_t check_dims(int dk, int dv, kda_dtype_t io) {
    if (dk <= 0 || dv <= 0) return fail(KDA_ERR_INVALID_ARG, "dk and dv must be positive");
    if (io != KDA_BF16 && io != KDA_F32) return fail(KDA_ERR_INVALID_ARG, "unknown io dtype");
    if (dk != dv) return fail(KDA_ERR_UNSUPPORTED, "dk != dv is not implemented");
    if (dk != 64 && dk != 128) return fail(KDA_ERR_UNSUPPORTED, "dk must be 64 or 128");
    return KDA_OK;
}

}  // namespace

extern "C" {

int kda_abi_version(void) { return KDA_ABI_VERSION; }

const char* kda_status_string(kda_status_t s) {
    switch (s) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_DECAY_RANGE: return "KDA_ERR_DECAY_RANGE";
        case KDA_ERR_NONFINITE: return "KDA_ERR_NONFINITE";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
    }
    return "KDA_ERR_UNKNOWN";
}

const char* kda_last_error_string(void) { return g_last_error; }

size_t kda_chunk_fwd_workspace_size(int B, int T, int H, int dk, int dv, kda_dtype_t io) {
    if (B < 0 || T < 0 || H < 0) return (size_t)-1;
    if (check_dims(dk, dv, io) != KDA_OK) return (size_t)-1;
    if ((long long)B * H >= (1LL << 31)) return (size_t)-1;
    // The tensor-core path balances sequences over the SMs through a state
    // handoff buffer; the fp32 path and empty problems need nothing.
    if (io != KDA_BF16 || T == 0 || (long long)B * H < 2) return 0;
    return kda::balanced_workspace_bytes((long long)B * H);
}

}  // extern "C"

// Scratch of kda_chunk_fwd_segmented_noalloc: 48 MB in the library's own
// device image, so that entry point allocates nothing. Every device that loads
// the library holds one instance until the process exits. It holds the
// (3 nseg - 2) 64 KB states per sequence of e.g. 48 sequences x 6 segments or
// 32 sequences x 8 segments.
static __device__ __align__(256) float g_seg_scratch[12u << 20];

namespace {

// Device address of g_seg_scratch, taken once per device (with that device
// current) on the first no-allocation call there. In host code the array's
// name is only a host-side stand-in, so kernels get this address instead.
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

cudaError_t seg_scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_seg_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

namespace {

// SMs of the current device, 0 if none is visible.
int device_sms() {
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        nsm <= 0) {
        cudaGetLastError();
        return 0;
    }
    return nsm;
}

// Device-planned split (nseg = 0): plans of up to min(32, chunks) segments;
// the workspace holds their states, then the decay probe (kPlanSamples chunks
// per batch row and head), then the plan {nseg, seg_chunks, lead}.
constexpr int kPlanSamples = 16;
int planned_max_segments(int T) {
    const int nch = (T + 63) / 64;
    return nch < kda::kPlanMaxSeg ? nch : kda::kPlanMaxSeg;
}
size_t probe_floats(int B, int H) { return ((size_t)B * kPlanSamples * H + 3) & ~(size_t)3; }
size_t planned_workspace_bytes(int B, int H, int nseg_max) {
    return (kda::segmented_workspace_floats((long long)B * H, nseg_max) + probe_floats(B, H)) * 4 + 16;
}

// The first segment's length in short segments for a split into nseg on nsm
// SMs: the cheapest of 1 .. 16 that leaves as many non-empty segments as an
// even split (so the workspace does not depend on the device); 1 without a
// device (nsm = 0).
int choose_lead(long long BH, int T, int nseg, int nsm, long long tl = -1) {
    using kda::split_cost;
    if (nseg <= 1 || nsm <= 0) return 1;
    int best = 1;
    long long best_cost = split_cost(BH, T, nseg, 1, nsm, tl);
    if (best_cost < 0) return 1;
    for (int lead = 2; lead <= 16; lead++) {
        const long long c = split_cost(BH, T, nseg, lead, nsm, tl);
        if (c >= 0 && c < best_cost) {
            best_cost = c;
            best = lead;
        }
    }
    return best;
}

kda_status_t chunk_fwd_impl(const void* q, const void* k, const void* v, const float* g,
                            const float* beta, const float* h0, void* o, float* hT, int B,
                            int T, int H, int dk, int dv, kda_dtype_t io, float* ckpt,
                            int ckpt_every, int* d_status, void* stream, int nseg = 1,
                            void* workspace = nullptr, size_t ws_bytes = 0,
                            bool check_only = false, void* bal_ws = nullptr,
                            size_t bal_bytes = 0, int lead_in = 0) {
    if (B < 0 || T < 0 || H < 0) return fail(KDA_ERR_INVALID_ARG, "B, T, H must be >= 0");
    kda_status_t st = check_dims(dk, dv, io);
    if (st != KDA_OK) return st;
    if ((long long)B * H >= (1LL << 31)) return fail(KDA_ERR_INVALID_ARG, "B*H too large");
    if (B == 0 || H == 0) return KDA_OK;
    const size_t esz = io == KDA_BF16 ? 2 : 4;
    size_t n_qk, n_v, n_b, n_s;
    if (!mul_ok(&n_qk, B, T, H, dk) || !mul_ok(&n_v, B, T, H, dv) || !mul_ok(&n_b, B, T, H) ||
        !mul_ok(&n_s, B, H, dk, dv))
        return fail(KDA_ERR_INVALID_ARG, "tensor size overflow");
    if (T > 0 && (!q || !k || !v || !g || !beta || !o))
        return fail(KDA_ERR_INVALID_ARG, "q, k, v, g, beta and o must be non-NULL");
    const void* ptrs[] = {q, k, v, g, h0, o, hT};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return fail(KDA_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    if (beta && !aligned4(beta)) return fail(KDA_ERR_INVALID_ARG, "beta must be 4-byte aligned");
    // o and hT are written while the inputs are still being read.
    const void* ins[] = {q, k, v, g, beta, h0};
    const size_t in_bytes[] = {n_qk * esz, n_qk * esz, n_v * esz, n_qk * 4, n_b * 4,
                               h0 ? n_s * 4 : 0};
    for (int i = 0; i < 6; i++) {
        if (overlaps(o, n_v * esz, ins[i], in_bytes[i]))
            return fail(KDA_ERR_INVALID_ARG, "o overlaps an input");
        if (i < 5 && overlaps(hT, n_s * 4, ins[i], in_bytes[i]))
            return fail(KDA_ERR_INVALID_ARG, "hT overlaps an input other than h0");
    }
    if (h0 && hT && h0 != hT && overlaps(hT, n_s * 4, h0, n_s * 4))
        return fail(KDA_ERR_INVALID_ARG, "hT partially overlaps h0");
    if (overlaps(o, n_v * esz, hT, n_s * 4)) return fail(KDA_ERR_INVALID_ARG, "o overlaps hT");
    if (ckpt) {
        if (ckpt_every <= 0 || ckpt_every % 64 != 0)
            return fail(KDA_ERR_INVALID_ARG, "ckpt_every must be a positive multiple of 64");
        if (!aligned16(ckpt)) return fail(KDA_ERR_INVALID_ARG, "ckpt must be 16-byte aligned");
        size_t n_c;
        if (!mul_ok(&n_c, n_s, (size_t)(T / ckpt_every)))
            return fail(KDA_ERR_INVALID_ARG, "tensor size overflow");
        const void* all[] = {q, k, v, g, beta, h0, o, hT};
        const size_t all_bytes[] = {n_qk * esz, n_qk * esz, n_v * esz, n_qk * 4, n_b * 4,
                                    h0 ? n_s * 4 : 0, n_v * esz, hT ? n_s * 4 : 0};
        for (int i = 0; i < 8; i++)
            if (overlaps(ckpt, n_c * 4, all[i], all_bytes[i]))
                return fail(KDA_ERR_INVALID_ARG, "ckpt overlaps another tensor");
    }

    int seg_chunks = 0, nseg_eff = 1, lead = 1;
    int nseg_max = 0;  // a device-planned split (nseg = 0): the largest plan
    if (nseg != 1) {
        if (io != KDA_BF16 || dk != 128)
            return fail(KDA_ERR_UNSUPPORTED, "segmented prefill needs bf16 and dk = dv = 128");
        const int nch = (T + 63) / 64;
        if (nseg == 0) {
            if (lead_in > 0)
                return fail(KDA_ERR_INVALID_ARG, "a device-planned split (nseg = 0) takes no lead");
            if (B > 65535) return fail(KDA_ERR_INVALID_ARG, "a device-planned split needs B <= 65535");
            nseg_max = planned_max_segments(T);
        } else if (nseg < 1 || (T > 0 && nseg > nch))
            return fail(KDA_ERR_INVALID_ARG, "nseg must be in 1 .. ceil(T / 64)");
        if (lead_in > 0 && T > 0 && lead_in > nch)
            return fail(KDA_ERR_INVALID_ARG, "lead must be <= 0 (the library's choice) or in 1 .. ceil(T / 64)");
        if (nseg > 0) {
            segment_shape(T, nseg, 1, &seg_chunks, &nseg_eff);
            lead = lead_in > 0 ? lead_in : choose_lead((long long)B * H, T, nseg_eff, device_sms());
            segment_shape(T, nseg_eff, lead, &seg_chunks, &nseg_eff);
        }
    }
    // Every argument but the workspace is valid.
    if (check_only) return KDA_OK;
    if (nseg_eff > 1 || nseg_max > 1) {
        const size_t need = nseg_max > 1
                                ? planned_workspace_bytes(B, H, nseg_max)
                                : kda::segmented_workspace_floats((long long)B * H, nseg_eff) * 4;
        if (!workspace || ws_bytes < need)
            return fail(KDA_ERR_WORKSPACE, "workspace smaller than the segmented size");
        if (!aligned16(workspace))
            return fail(KDA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
        const void* all[] = {q, k, v, g, beta, h0, o, hT};
        const size_t all_bytes[] = {n_qk * esz, n_qk * esz, n_v * esz, n_qk * 4, n_b * 4,
                                    h0 ? n_s * 4 : 0, n_v * esz, hT ? n_s * 4 : 0};
        for (int i = 0; i < 8; i++)
            if (overlaps(workspace, need, all[i], all_bytes[i]))
                return fail(KDA_ERR_INVALID_ARG, "workspace overlaps another tensor");
    }

    kda::ChunkFwdArgs a{q, k, v, g, beta, h0, o, hT, B, T, H, dk, dv, d_status,
                        static_cast<cudaStream_t>(stream)};
    a.ckpt = ckpt;
    a.ckpt_every = ckpt ? ckpt_every : 0;
    // A prefill workspace of the queried size enables the balanced schedule;
    // without one (or a smaller one) every sequence gets its own CTA.
    if (bal_ws && nseg_eff <= 1 && io == KDA_BF16) {
        const size_t need = kda::balanced_workspace_bytes((long long)B * H);
        if (bal_bytes < need) {
            bal_ws = nullptr;
        } else {
            if (!aligned16(bal_ws))
                return fail(KDA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
            const void* all[] = {q, k, v, g, beta, h0, o, hT};
            const size_t all_bytes[] = {n_qk * esz, n_qk * esz, n_v * esz, n_qk * 4, n_b * 4,
                                        h0 ? n_s * 4 : 0, n_v * esz, hT ? n_s * 4 : 0};
            for (int i = 0; i < 8; i++)
                if (overlaps(bal_ws, need, all[i], all_bytes[i]))
                    return fail(KDA_ERR_INVALID_ARG, "workspace overlaps another tensor");
        }
        a.bal_ws = bal_ws;
    }
    cudaError_t e;
    if (nseg_max > 1) {
        // probe -> plan -> segment pass, scan, correction: all on the stream
        const long long BH = (long long)B * H;
        float* wsf = static_cast<float*>(workspace);
        float* probe = wsf + kda::segmented_workspace_floats(BH, nseg_max);
        int* plan = reinterpret_cast<int*>(probe + probe_floats(B, H));
        e = kda::launch_decay_probe(g, B, T, H, dk, kPlanSamples, probe, a.stream);
        if (e == cudaSuccess)
            e = kda::launch_segment_plan(probe, B * kPlanSamples * H, BH, T, device_sms(),
                                         nseg_max, plan, a.stream);
        if (e == cudaSuccess) e = kda::launch_chunk_fwd_tc_segmented_planned(a, nseg_max, wsf, plan);
    } else {
        e = nseg_eff > 1 ? kda::launch_chunk_fwd_tc_segmented(a, nseg_eff, seg_chunks, lead,
                                                              static_cast<float*>(workspace))
            : io == KDA_BF16 ? kda::launch_chunk_fwd_tc(a)
                             : kda::launch_chunk_fwd_simt(a, io);
    }
    if (e != cudaSuccess) {
        set_last_error(cudaGetErrorString(e));
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

}  // namespace

extern "C" {

kda_status_t kda_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                           const float* beta, const float* h0, void* o, float* hT, int B,
                           int T, int H, int dk, int dv, kda_dtype_t io, void* workspace,
                           size_t ws_bytes, int* d_status, void* stream) {
    NvtxRange nvtx_range("kda_chunk_fwd");
    return chunk_fwd_impl(q, k, v, g, beta, h0, o, hT, B, T, H, dk, dv, io, nullptr, 0,
                          d_status, stream, 1, nullptr, 0, false, workspace, ws_bytes);
}

kda_status_t kda_chunk_fwd_ckpt(const void* q, const void* k, const void* v, const float* g,
                                const float* beta, const float* h0, void* o, float* hT,
                                float* ckpt, int ckpt_every, int B, int T, int H, int dk, int dv,
                                kda_dtype_t io, int* d_status, void* stream) {
    NvtxRange nvtx_range("kda_chunk_fwd_ckpt");
    if (!ckpt) return fail(KDA_ERR_INVALID_ARG, "ckpt must be non-NULL");
    return chunk_fwd_impl(q, k, v, g, beta, h0, o, hT, B, T, H, dk, dv, io, ckpt, ckpt_every,
                          d_status, stream);
}

int kda_chunk_fwd_segments_hint(int B, int T, int H, int dk, int dv, kda_dtype_t io) {
    if (B < 0 || T < 0 || H < 0 || check_dims(dk, dv, io) != KDA_OK) return -1;
    if ((long long)B * H >= (1LL << 31)) return -1;
    if (io != KDA_BF16 || dk != 128 || B == 0 || H == 0) return 1;
    const int nsm = device_sms();
    if (nsm <= 0) return 1;
    const long long BH = (long long)B * H;
    // Whole segments for every run: the data is not known here.
    long long cost[kda::kPlanCosts];
    kda::fill_plan_costs(BH, T, nsm, -1, cost);
    return kda::choose_plan(BH, T, nsm, kda::kPlanMaxSeg, cost).nseg;
}

int kda_chunk_fwd_segments_hint_decay(int B, int T, int H, int dk, int dv, kda_dtype_t io,
                                                                        const float* probe, int nprobe, int* lead) {
    if (B < 0 || T < 0 || H < 0 || check_dims(dk, dv, io) != KDA_OK) return -1;
    if ((long long)B * H >= (1LL << 31)) return -1;
    if (nprobe < 0 || (nprobe > 0 && !probe)) return -1;
    if (lead) *lead = 1;
    if (io != KDA_BF16 || dk != 128 || B == 0 || H == 0) return 1;
    const int nsm = device_sms();
    if (nsm <= 0) return 1;
    // The weakest decay per chunk the sample shows (no entries, or a
    // non-finite one: unknown, so whole segments).
    float cd = nprobe > 0 ? -INFINITY : 0.f;
    for (int i = 0; i < nprobe; i++) {
        if (!std::isfinite(probe[i])) {
            cd = 0.f;
            break;
        }
        cd = std::max(cd, probe[i]);
    }
    const long long BH = (long long)B * H, tl = kda::transition_chunks(cd, T);
    long long cost[kda::kPlanCosts];
    kda::fill_plan_costs(BH, T, nsm, tl, cost);
    const kda::SegPlan plan = kda::choose_plan(BH, T, nsm, kda::kPlanMaxSeg, cost);
    if (lead) *lead = plan.lead;
    return plan.nseg;
}

kda_status_t kda_chunk_fwd_decay_probe(const float* g, int B, int T, int H, int dk, int nsample,
                                       float* d_probe, void* stream) {
    NvtxRange nvtx_range("kda_chunk_fwd_decay_probe");
    if (B < 0 || T < 0 || H < 0) return fail(KDA_ERR_INVALID_ARG, "B, T, H must be >= 0");
    if (dk != 64 && dk != 128) return fail(KDA_ERR_UNSUPPORTED, "dk must be 64 or 128");
    if (nsample < 1 || nsample > 4096) return fail(KDA_ERR_INVALID_ARG, "nsample must be in 1 .. 4096");
    if ((long long)B * H >= (1LL << 31) || B > 65535 || H > 8 * 65535)
        return fail(KDA_ERR_INVALID_ARG, "B must be <= 65535, H <= 524280 and B*H < 2^31");
    if (B == 0 || H == 0 || T == 0) return KDA_OK;
    size_t n_g, n_p;
    if (!mul_ok(&n_g, B, T, H, dk) || !mul_ok(&n_p, B, nsample, H))
        return fail(KDA_ERR_INVALID_ARG, "tensor size overflow");
    if (!g || !d_probe) return fail(KDA_ERR_INVALID_ARG, "g and d_probe must be non-NULL");
    if (!aligned16(g) || !aligned4(d_probe))
        return fail(KDA_ERR_INVALID_ARG, "g must be 16-byte and d_probe 4-byte aligned");
    if (overlaps(d_probe, n_p * 4, g, n_g * 4))
        return fail(KDA_ERR_INVALID_ARG, "d_probe overlaps g");
    cudaError_t e = kda::launch_decay_probe(g, B, T, H, dk, nsample, d_probe,
                                            static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        set_last_error(cudaGetErrorString(e));
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

int kda_chunk_fwd_segment_plan(int B, int T, int H, int dk, int dv, kda_dtype_t io, int nseg,
                               int lead_in, int* seg_chunks, int* lead) {
    if (B < 0 || T < 0 || H < 0 || check_dims(dk, dv, io) != KDA_OK) return -1;
    if ((long long)B * H >= (1LL << 31)) return -1;
    const int nch = (T + 63) / 64;
    if (nseg < 1 || (T > 0 && nseg > nch)) return -1;
    if (nseg > 1 && (io != KDA_BF16 || dk != 128)) return -1;
    if (nseg > 1 && lead_in > 0 && T > 0 && lead_in > nch) return -1;
    int sc = nch, se = 1, ld = 1;
    if (nseg > 1) {
        segment_shape(T, nseg, 1, &sc, &se);
        ld = lead_in > 0 ? lead_in : choose_lead((long long)B * H, T, se, device_sms());
        segment_shape(T, se, ld, &sc, &se);
    }
    if (seg_chunks) *seg_chunks = se > 1 ? sc : nch;
    if (lead) *lead = ld;
    return se;
}

size_t kda_chunk_fwd_segmented_workspace_size(int B, int T, int H, int dk, int dv,
                                              kda_dtype_t io, int nseg) {
    if (B < 0 || T < 0 || H < 0 || check_dims(dk, dv, io) != KDA_OK) return (size_t)-1;
    if ((long long)B * H >= (1LL << 31)) return (size_t)-1;
    const int nch = (T + 63) / 64;
    if (nseg != 1 && (io != KDA_BF16 || dk != 128)) return (size_t)-1;
    if (nseg == 0) {  // planned on the device
        if (B > 65535) return (size_t)-1;
        const int nmax = planned_max_segments(T);
        return nmax > 1 && B > 0 && H > 0 ? planned_workspace_bytes(B, H, nmax) : 0;
    }
    if (nseg < 1 || (T > 0 && nseg > nch)) return (size_t)-1;
    int sc, se;
    segment_shape(T, nseg, 1, &sc, &se);
    return se > 1 ? kda::segmented_workspace_floats((long long)B * H, se) * 4 : 0;
}

kda_status_t kda_chunk_fwd_segmented(const void* q, const void* k, const void* v,
                                     const float* g, const float* beta, const float* h0, void* o,
                                     float* hT, int B, int T, int H, int dk, int dv,
                                     kda_dtype_t io, int nseg, int lead, void* workspace,
                                     size_t ws_bytes, int* d_status, void* stream) {
    NvtxRange nvtx_range("kda_chunk_fwd_segmented");
    return chunk_fwd_impl(q, k, v, g, beta, h0, o, hT, B, T, H, dk, dv, io, nullptr, 0, d_status,
                          stream, nseg, workspace, ws_bytes, false, nullptr, 0, lead);
}

kda_status_t kda_chunk_fwd_segmented_noalloc(const void* q, const void* k, const void* v,
                                             const float* g, const float* beta, const float* h0,
                                             void* o, float* hT, int B, int T, int H, int dk,
                                             int dv, kda_dtype_t io, int nseg, int lead,
                                             int* d_status, void* stream) {
    NvtxRange nvtx_range("kda_chunk_fwd_segmented_noalloc");
    // Argument errors first, as for the other entry points.
    kda_status_t st = chunk_fwd_impl(q, k, v, g, beta, h0, o, hT, B, T, H, dk, dv, io, nullptr,
                                     0, d_status, stream, nseg, nullptr, 0, /*check_only=*/true,
                                     nullptr, 0, lead);
    if (st != KDA_OK) return st;
    const size_t need = kda_chunk_fwd_segmented_workspace_size(B, T, H, dk, dv, io, nseg);
    if (need > sizeof(g_seg_scratch))
        return fail(KDA_ERR_WORKSPACE, "problem needs more than the 48 MB static segment scratch");
    void* ws = nullptr;
    if (need > 0) {
        cudaError_t e = seg_scratch_address(&ws);
        if (e != cudaSuccess) {
            set_last_error(cudaGetErrorString(e));
            return KDA_ERR_CUDA;
        }
    }
    return chunk_fwd_impl(q, k, v, g, beta, h0, o, hT, B, T, H, dk, dv, io, nullptr, 0, d_status,
                          stream, nseg, ws, need > 0 ? sizeof(g_seg_scratch) : 0, false, nullptr,
                          0, lead);
}

namespace {

// Common checks of the two whole-slice passes: bf16, dk = dv = 128, inputs
// present and aligned, `state` and `o` (either may be absent) clear of the
// inputs and of each other.
kda_status_t slice_args(const void* q, const void* k, const float* g, const float* beta,
                        const void* state, size_t state_bytes, const void* o, int B, int T, int H,
                        int dk, int dv, kda_dtype_t io, size_t* n_qk_out) {
    if (B < 0 || T < 0 || H < 0) return fail(KDA_ERR_INVALID_ARG, "B, T, H must be >= 0");
    kda_status_t st = check_dims(dk, dv, io);
    if (st != KDA_OK) return st;
    if (io != KDA_BF16 || dk != 128)
        return fail(KDA_ERR_UNSUPPORTED, "slice passes need bf16 and dk = dv = 128");
    if ((long long)B * H >= (1LL << 31)) return fail(KDA_ERR_INVALID_ARG, "B*H too large");
    size_t n_qk, n_b, n_s;
    if (!mul_ok(&n_qk, B, T, H, dk) || !mul_ok(&n_b, B, T, H) || !mul_ok(&n_s, B, H, dk, dv))
        return fail(KDA_ERR_INVALID_ARG, "tensor size overflow");
    if (B == 0 || H == 0) return KDA_OK;
    if (T > 0 && (!q || !k || !g || !beta))
        return fail(KDA_ERR_INVALID_ARG, "q, k, g and beta must be non-NULL");
    if (!state) return fail(KDA_ERR_INVALID_ARG, "the state tensor must be non-NULL");
    const void* ptrs[] = {q, k, g, state, o};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return fail(KDA_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    if (beta && !aligned4(beta)) return fail(KDA_ERR_INVALID_ARG, "beta must be 4-byte aligned");
    const void* ins[] = {q, k, g, beta};
    const size_t in_bytes[] = {n_qk * 2, n_qk * 2, n_qk * 4, n_b * 4};
    const size_t o_bytes = n_qk * 2;  // dv = dk
    for (int i = 0; i < 4; i++) {
        if (overlaps(state, state_bytes, ins[i], in_bytes[i]))
            return fail(KDA_ERR_INVALID_ARG, "the state tensor overlaps an input");
        if (overlaps(o, o_bytes, ins[i], in_bytes[i]))
            return fail(KDA_ERR_INVALID_ARG, "o overlaps an input");
    }
    if (overlaps(o, o_bytes, state, state_bytes))
        return fail(KDA_ERR_INVALID_ARG, "o overlaps the state tensor");
    *n_qk_out = n_qk;
    return KDA_OK;
}

}  // namespace

kda_status_t kda_chunk_fwd_slice_transition(const void* q, const void* k, const float* g,
                                            const float* beta, float* M, int B, int T, int H,
                                            int dk, kda_dtype_t io, int* d_status,
                                            void* stream) {
    NvtxRange nvtx_range("kda_chunk_fwd_slice_transition");
    size_t n_qk = 0, n_m = 0;
    if (B >= 0 && H >= 0 && dk > 0) mul_ok(&n_m, (size_t)B, (size_t)H, (size_t)dk, (size_t)dk);
    kda_status_t st = slice_args(q, k, g, beta, M, n_m * 4, nullptr, B, T, H, dk, dk, io, &n_qk);
    if (st != KDA_OK || B == 0 || H == 0) return st;
    // v is not read (the run has v = 0); q stands in for its tensor map.
    kda::ChunkFwdArgs a{q, k, q, g, beta, nullptr, nullptr, nullptr, B, T, H, dk, dk, d_status,
                        static_cast<cudaStream_t>(stream)};
    cudaError_t e = kda::launch_chunk_fwd_tc_slice(a, 1, M);
    if (e != cudaSuccess) {
        set_last_error(cudaGetErrorString(e));
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

kda_status_t kda_chunk_fwd_slice_correct(const void* q, const void* k, const float* g,
                                         const float* beta, const float* S_in, void* o, int B,
                                         int T, int H, int dk, int dv, kda_dtype_t io,
                                         int* d_status, void* stream) {
    NvtxRange nvtx_range("kda_chunk_fwd_slice_correct");
    size_t n_qk = 0, n_s = 0;
    if (B >= 0 && H >= 0 && dk > 0 && dv > 0)
        mul_ok(&n_s, (size_t)B, (size_t)H, (size_t)dk, (size_t)dv);
    kda_status_t st = slice_args(q, k, g, beta, S_in, n_s * 4, o, B, T, H, dk, dv, io, &n_qk);
    if (st != KDA_OK || B == 0 || H == 0 || T == 0) return st;
    if (!o) return fail(KDA_ERR_INVALID_ARG, "o must be non-NULL");
    kda::ChunkFwdArgs a{q, k, q, g, beta, nullptr, o, nullptr, B, T, H, dk, dv, d_status,
                        static_cast<cudaStream_t>(stream)};
    cudaError_t e = kda::launch_chunk_fwd_tc_slice(a, 2, const_cast<float*>(S_in));
    if (e != cudaSuccess) {
        set_last_error(cudaGetErrorString(e));
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

kda_status_t kda_state_scan(const float* s0, const float* m, float* x_in, float* hT, int nslice,
                            int B, int H, int dk, int dv, void* stream) {
    NvtxRange nvtx_range("kda_state_scan");
    if (nslice < 1 || B < 0 || H < 0)
        return fail(KDA_ERR_INVALID_ARG, "nslice must be >= 1, B and H >= 0");
    if (dk <= 0 || dv <= 0) return fail(KDA_ERR_INVALID_ARG, "dk and dv must be positive");
    if (dk != 128 || dv != 128) return fail(KDA_ERR_UNSUPPORTED, "the scan needs dk = dv = 128");
    if ((long long)B * H >= (1LL << 31)) return fail(KDA_ERR_INVALID_ARG, "B*H too large");
    if (B == 0 || H == 0) return KDA_OK;
    size_t n_s, n_all, n_rest;
    if (!mul_ok(&n_s, B, H, dk, dv) || !mul_ok(&n_all, n_s, (size_t)nslice) ||
        !mul_ok(&n_rest, n_s, (size_t)(nslice - 1)))
        return fail(KDA_ERR_INVALID_ARG, "tensor size overflow");
    if (!s0 || (nslice > 1 && (!m || !x_in)))
        return fail(KDA_ERR_INVALID_ARG, "s0, and for nslice > 1 m and x_in, must be non-NULL");
    const void* ptrs[] = {s0, m, x_in, hT};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return fail(KDA_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    if (overlaps(x_in, n_rest * 4, s0, n_all * 4) || overlaps(x_in, n_rest * 4, m, n_rest * 4) ||
        overlaps(hT, n_s * 4, s0, n_all * 4) || overlaps(hT, n_s * 4, m, n_rest * 4) ||
        overlaps(hT, n_s * 4, x_in, n_rest * 4))
        return fail(KDA_ERR_INVALID_ARG, "outputs overlap the inputs or each other");
    cudaError_t e = kda::launch_slice_scan(s0, m, x_in, hT, B * H, nslice,
                                           static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        set_last_error(cudaGetErrorString(e));
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

kda_status_t kda_selftest_wait_timeout(long long clocks, int* d_status, void* stream) {
    NvtxRange nvtx_range("kda_selftest_wait_timeout");
    if (clocks <= 0 || clocks > (1LL << 31))
        return fail(KDA_ERR_INVALID_ARG, "clocks must be in 1 .. 2^31");
    if (!d_status || ((uintptr_t)d_status & 3))
        return fail(KDA_ERR_INVALID_ARG, "d_status must be a non-NULL, 4-byte aligned int");
    cudaError_t e = kda::launch_selftest_wait(clocks, d_status, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        set_last_error(cudaGetErrorString(e));
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

kda_status_t kda_decode_step(const void* q, const void* k, const void* v, const float* g,
                             const float* beta, float* S, void* o, int N, int H, int dk,
                             int dv, kda_dtype_t io, int* d_status, void* stream) {
    NvtxRange nvtx_range("kda_decode_step");
    if (N < 0 || H < 0) return fail(KDA_ERR_INVALID_ARG, "N and H must be >= 0");
    kda_status_t st = check_dims(dk, dv, io);
    if (st != KDA_OK) return st;
    // two blocks per (sequence, head)
    if ((long long)N * H * 2 >= (1LL << 31)) return fail(KDA_ERR_INVALID_ARG, "N*H too large");
    if (N == 0 || H == 0) return KDA_OK;
    if (!q || !k || !v || !g || !beta || !S || !o)
        return fail(KDA_ERR_INVALID_ARG, "all decode pointers must be non-NULL");
    const void* ptrs[] = {q, k, v, g, S, o};
    for (const void* p : ptrs)
        if (!aligned16(p)) return fail(KDA_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    if (!aligned4(beta)) return fail(KDA_ERR_INVALID_ARG, "beta must be 4-byte aligned");
    const size_t esz = io == KDA_BF16 ? 2 : 4;
    size_t n_k, n_v, n_s;
    if (!mul_ok(&n_k, N, H, dk) || !mul_ok(&n_v, N, H, dv) || !mul_ok(&n_s, N, H, dk, dv))
        return fail(KDA_ERR_INVALID_ARG, "tensor size overflow");
    const void* ins[] = {q, k, v, g, beta};
    const size_t in_bytes[] = {n_k * esz, n_k * esz, n_v * esz, n_k * 4, (size_t)N * H * 4};
    for (int i = 0; i < 5; i++) {
        if (overlaps(o, n_v * esz, ins[i], in_bytes[i]) || overlaps(S, n_s * 4, ins[i], in_bytes[i]))
            return fail(KDA_ERR_INVALID_ARG, "o or S overlaps an input");
    }
    if (overlaps(o, n_v * esz, S, n_s * 4)) return fail(KDA_ERR_INVALID_ARG, "o overlaps S");
    kda::DecodeArgs a{q, k, v, g, beta, S, o, N, H, dk, dv, d_status,
                      static_cast<cudaStream_t>(stream)};
    cudaError_t e = kda::launch_decode(a, io);
    if (e != cudaSuccess) {
        set_last_error(cudaGetErrorString(e));
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

kda_status_t kda_decode_multi(const void* q, const void* k, const void* v, const float* g,
                              const float* beta, float* S, void* o, const int* ntok, int N, int K,
                              int H, int dk, int dv, kda_dtype_t io, int commit, int* d_status,
                              void* stream) {
    NvtxRange nvtx_range("kda_decode_multi");
    if (N < 0 || H < 0 || K < 0) return fail(KDA_ERR_INVALID_ARG, "N, K and H must be >= 0");
    kda_status_t st = check_dims(dk, dv, io);
    if (st != KDA_OK) return st;
    if ((long long)N * H >= (1LL << 31)) return fail(KDA_ERR_INVALID_ARG, "N*H too large");
    if (N == 0 || H == 0 || K == 0) return KDA_OK;
    if (!q || !k || !v || !g || !beta || !S)
        return fail(KDA_ERR_INVALID_ARG, "q, k, v, g, beta and S must be non-NULL");
    if (!o && !commit) return fail(KDA_ERR_INVALID_ARG, "verify (commit = 0) needs o");
    const void* ptrs[] = {q, k, v, g, S, o};
    for (const void* p : ptrs)
        if (p && !aligned16(p)) return fail(KDA_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    if (!aligned4(beta) || (ntok && !aligned4(ntok)))
        return fail(KDA_ERR_INVALID_ARG, "beta and ntok must be 4-byte aligned");
    const size_t esz = io == KDA_BF16 ? 2 : 4;
    size_t n_k, n_v, n_b, n_s;
    if (!mul_ok(&n_k, N, K, H, dk) || !mul_ok(&n_v, N, K, H, dv) || !mul_ok(&n_b, N, K, H) ||
        !mul_ok(&n_s, N, H, dk, dv))
        return fail(KDA_ERR_INVALID_ARG, "tensor size overflow");
    const void* ins[] = {q, k, v, g, beta, ntok};
    const size_t in_bytes[] = {n_k * esz, n_k * esz, n_v * esz, n_k * 4, n_b * 4,
                               ntok ? (size_t)N * 4 : 0};
    for (int i = 0; i < 6; i++) {
        if (overlaps(o, n_v * esz, ins[i], in_bytes[i]) || overlaps(S, n_s * 4, ins[i], in_bytes[i]))
            return fail(KDA_ERR_INVALID_ARG, "o or S overlaps an input");
    }
    if (overlaps(o, n_v * esz, S, n_s * 4)) return fail(KDA_ERR_INVALID_ARG, "o overlaps S");
    kda::MultiDecodeArgs a{q, k, v, g, beta, S, o, ntok, N, K, H, dk, dv, commit ? 1 : 0,
                           d_status, static_cast<cudaStream_t>(stream)};
    cudaError_t e = kda::launch_decode_multi(a, io);
    if (e != cudaSuccess) {
        set_last_error(cudaGetErrorString(e));
        return KDA_ERR_CUDA;
    }
    return KDA_OK;
}

}  // extern "C"
