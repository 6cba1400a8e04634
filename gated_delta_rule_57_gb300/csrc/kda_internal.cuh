// Internal declarations shared by the KDA CUDA translation units.
// Not part of the public ABI (include/kda.h is).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// Launch parameters common to both chunked-forward paths. Pointers are device
// pointers; layouts as documented in kda.h.
struct ChunkFwdArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    const float* beta;
    const float* h0;  // may be null
    void* o;
    float* hT;  // may be null
    int B, T, H, dk, dv;
    int* d_status;  // may be null
    cudaStream_t stream;
    float* ckpt = nullptr;  // [B, H, T / ckpt_every, dk, dv] or null
    int ckpt_every = 0;     // tokens between checkpoints (multiple of 64)
    // balanced_workspace_bytes(B * H) bytes for the balanced schedule of the
    // tensor-core prefill, or null (one CTA per sequence)
    void* bal_ws = nullptr;
};

struct DecodeArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    const float* beta;
    float* S;
    void* o;
    int N, H, dk, dv;
    int* d_status;
    cudaStream_t stream;
};

struct MultiDecodeArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    const float* beta;
    float* S;
    void* o;          // may be null when commit != 0
    const int* ntok;  // may be null: every sequence takes all K tokens
    int N, K, H, dk, dv;
    int commit;
    int* d_status;
    cudaStream_t stream;
};

// Each launcher returns cudaSuccess or the launch error.
cudaError_t launch_chunk_fwd_simt(const ChunkFwdArgs& a, kda_dtype_t io);
cudaError_t launch_chunk_fwd_tc(const ChunkFwdArgs& a);
// Long sequences split in time into nseg segments (bf16, dk = dv = 128):
// the first lead * seg_chunks 64-token chunks long, the others seg_chunks;
// segment pass, prefix scan, correction pass. ws holds
// segmented_workspace_floats(B * H, nseg) floats.
cudaError_t launch_chunk_fwd_tc_segmented(const ChunkFwdArgs& a, int nseg, int seg_chunks,
                                          int lead, float* ws);
cudaError_t launch_segment_scan(const float* s0, const float* m, float* sin, float* hT, int BH,
                                int nseg, cudaStream_t stream);
cudaError_t launch_segment_scan_planned(const float* s0, const float* m, float* sin, float* hT,
                                        int BH, int nseg_max, const int* plan,
                                        cudaStream_t stream);
// One time slice of every sequence (bf16, dk = dv = 128), for a sequence
// split across devices: which = 1 writes the slice's transition (the run
// from the identity with v = 0) to state [B*H][dk][dk]; which = 2 runs from
// the incoming states `state` [B*H][dk][dv] with v = 0 and adds its outputs
// to o. a.v is not read.
cudaError_t launch_chunk_fwd_tc_slice(const ChunkFwdArgs& a, int which, float* state);
// Scan over nslice slices stored slice-major: s0 [nslice][BH], m [nslice - 1][BH]
// (the transitions of slices 1..), sin [nslice - 1][BH] (incoming states of
// slices 1..), hT [BH] (nullable).
cudaError_t launch_slice_scan(const float* s0, const float* m, float* sin, float* hT, int BH,
                              int nslice, cudaStream_t stream);
// Sampled decay bound for planning a split in time: out[b][s][h] = sum over
// the tokens of chunk floor(s * nch / nsample) of max over channels of
// g[b][t][h][:] (g [B][T][H][dk] fp32, dk = 64 or 128).
cudaError_t launch_decay_probe(const float* g, int B, int T, int H, int dk, int nsample,
                               float* out, cudaStream_t stream);
// Handoff buffer of the balanced prefill schedule: one 128 x 128 fp32 state
// and one int flag per sequence (flags rounded up to 256 bytes).
inline size_t balanced_workspace_bytes(long long BH) {
    return (size_t)BH * 128u * 128u * 4u + (((size_t)BH * 4u + 255u) & ~(size_t)255u);
}
inline size_t segmented_workspace_floats(long long BH, int nseg) {
    // per sequence: nseg zero-start final states, nseg - 1 transitions and
    // nseg - 1 incoming states, 128 x 128 fp32 each
    return (size_t)BH * (size_t)(3 * nseg - 2) * 128u * 128u;
}
// ---- Planning a split in time (shared by the host hints and the planning
// kernel, so both choose the same split).
constexpr int kPlanMaxSeg = 32;   // segment counts considered: 2 .. 32
constexpr int kPlanMaxLead = 16;  // first-segment lengths considered: 1 .. 16
//
// Segments of a sequence of nch = ceil(T / 64) chunks split into nseg:
// segment 0 spans lead * sc chunks, every later one sc = ceil(nch / (lead +
// nseg - 1)); *nseg_eff is the number of non-empty segments that gives (at
// most nseg): the least count whose lengths reach nch.
__host__ __device__ inline void segment_shape(int T, int nseg, int lead, int* seg_chunks,
                                              int* nseg_eff) {
    const int nch = (T + 63) / 64;
    const int sc = nch > 0 ? (nch + lead + nseg - 2) / (lead + nseg - 1) : 1;
    int ne = (nch + sc - 1) / sc - lead + 1;
    ne = ne < 1 ? 1 : (ne > nseg ? nseg : ne);
    *seg_chunks = sc;
    *nseg_eff = ne;
}

// Chunk steps on the critical path of a split run with one CTA per SM. The
// segment pass starts the BH long first segments, the other SMs take the
// 2 BH (nseg - 1) short runs (segments from zero and transitions) and every
// SM joins once the long runs end; the correction pass has BH (nseg - 1)
// short runs. tl < 0: the runs with v = 0 (transitions, corrections) take
// their whole segment; else about tl chunks (they stop once their state is
// exactly zero). Returns -1 when the split leaves empty segments.
template <typename I>
__host__ __device__ inline I split_cost_t(I BH, int T, int nseg, int lead, int nsm, I tl) {
    int sc, se;
    segment_shape(T, nseg, lead, &sc, &se);
    if (se != nseg) return -1;
    const I n = nsm;
    auto waves = [&](I ctas) { return (ctas + n - 1) / n; };
    if (tl >= 0 && tl < sc) {
        // The BH (nseg - 1) segments from zero run sc chunks each, the
        // transitions (dispatched after them) and corrections about tl.
        const I z = BH * (nseg - 1);
        I p1;
        if (BH >= n) {
            p1 = waves(BH) * lead * sc + waves(z) * (sc + tl);
        } else {
            const I free_sms = n - BH, wz = (z + free_sms - 1) / free_sms;
            const I a = (I)lead * sc, b = wz * (sc + tl);
            p1 = wz <= lead ? (a > b ? a : b)
                            : ((I)lead + waves(z - free_sms * lead)) * sc + waves(z) * tl;
        }
        return p1 + waves(z) * tl;
    }
    const I shorts = 2 * BH * (nseg - 1);
    I p1;
    if (BH >= n) {
        p1 = waves(BH) * lead * sc + waves(shorts) * sc;
    } else {
        const I free_sms = n - BH;
        const I w = (shorts + free_sms - 1) / free_sms;
        p1 = w <= lead ? (I)lead * sc : ((I)lead + waves(shorts - free_sms * lead)) * sc;
    }
    return p1 + waves(BH * (nseg - 1)) * sc;
}
__host__ __device__ inline long long split_cost(long long BH, int T, int nseg, int lead, int nsm,
                                                long long tl = -1) {
    return split_cost_t<long long>(BH, T, nseg, lead, nsm, tl);
}
// True when every value split_cost forms for these sizes (s <= 32 segments,
// leads <= 16, tl <= chunks) fits in 32 bits, so split_cost_t<int> gives the
// same costs.
__host__ __device__ inline bool plan_fits_32(long long BH, int T, int nsm) {
    const long long nch = (T + 63) / 64;
    if (nsm <= 0 || BH >= (1LL << 24) || nch >= (1LL << 24)) return false;
    const long long waves_max = (BH * 2 * kPlanMaxSeg + nsm - 1) / nsm + kPlanMaxLead + 2;
    return waves_max * (2 * nch + 2) * 4 < (1LL << 31);
}


// Transition length (chunks) to count on for a probe statistic cd (the
// largest sum over a chunk of the per-token max log-decay; see
// kda_chunk_fwd_decay_probe): a state shrinks at least by e^cd per chunk and
// is exactly zero past 2^-149 = e^-103.28, one chunk later the run has
// stopped. cd >= 0 or not finite: -1 (whole segments).
__host__ __device__ inline long long transition_chunks(float cd, int T) {
    if (!(cd < 0.f)) return -1;
    const long long nch = (T + 63) / 64;
    const long long t = 2 + (long long)ceilf(103.28f / -cd);
    return t < nch ? t : nch;
}

// The plan: the segment count of 2 .. min(32, nch, nseg_max) with the fewest
// chunk steps on the critical path (each at its best first-segment length of
// 1 .. 16, plus one step per scan step), a larger count taken only when it
// saves 2 %, and no split (1) unless it saves a fifth against whole
// sequences. cost[s * kPlanStride + l] = split_cost for s segments and lead l
// (filled for s = 2 .. 32, l = 1 .. 16; see fill_plan_costs).
struct SegPlan {
    int nseg, seg_chunks, lead;
};
constexpr int kPlanStride = kPlanMaxLead + 1;
constexpr int kPlanCosts = (kPlanMaxSeg + 1) * kPlanStride;
// For s segments: the cheapest first-segment length (the first of equal
// costs), from row[l] = cost with lead l; -1 when lead 1 leaves empty segments.
__host__ __device__ inline void best_lead(const long long* row, long long* cost, int* lead) {
    int ld = 1;
    long long c = row[1];
    if (c >= 0) {
        for (int l = 2; l <= kPlanMaxLead; l++) {
            if (row[l] >= 0 && row[l] < c) {
                c = row[l];
                ld = l;
            }
        }
    }
    *cost = c;
    *lead = ld;
}
// The choice over segment counts from each count's best (cost, lead):
// bc[s], bl[s] for s = 2 .. 32.
__host__ __device__ inline SegPlan choose_plan_best(long long BH, int T, int nsm, int nseg_max,
                                                    const long long* bc, const int* bl) {
    const long long nch = (T + 63) / 64;
    SegPlan plan{1, (int)(nch > 0 ? nch : 1), 1};
    if (nsm <= 0 || BH <= 0 || nch < 2) return plan;
    const long long base = ((BH + nsm - 1) / nsm) * nch;
    int best = 1, best_lead = 1;
    long long best_cost = -1;
    for (int s = 2; s <= kPlanMaxSeg && s <= nch && s <= nseg_max; s++) {
        // (a count whose even split leaves empty segments costs -1 at lead 1)
        const int ld = bl[s];
        const long long c = bc[s];
        if (c < 0) continue;
        const long long total = c + (s - 1);
        if (best_cost < 0 || total * 50 < best_cost * 49) {
            best_cost = total;
            best = s;
            best_lead = ld;
        }
    }
    if (!(best_cost >= 0 && best_cost * 5 < base * 4)) return plan;
    plan.nseg = best;
    plan.lead = best_lead;
    int se;
    segment_shape(T, best, best_lead, &plan.seg_chunks, &se);
    return plan;
}
// The same from the whole cost table (cost[s * kPlanStride + l]).
__host__ __device__ inline SegPlan choose_plan(long long BH, int T, int nsm, int nseg_max,
                                               const long long* cost) {
    long long bc[kPlanMaxSeg + 1];
    int bl[kPlanMaxSeg + 1];
    for (int s = 0; s <= kPlanMaxSeg; s++) best_lead(cost + s * kPlanStride, &bc[s], &bl[s]);
    return choose_plan_best(BH, T, nsm, nseg_max, bc, bl);
}

// Host side: the whole cost table, one entry at a time (nsm > 0).
inline void fill_plan_costs(long long BH, int T, int nsm, long long tl, long long* cost) {
    for (int s = 0; s <= kPlanMaxSeg; s++)
        for (int l = 0; l <= kPlanMaxLead; l++)
            cost[s * kPlanStride + l] = (s >= 2 && l >= 1) ? split_cost(BH, T, s, l, nsm, tl) : -1;
}

// Device-planned split (kda_chunk_fwd_segmented with nseg = 0): the planning
// kernel reduces a decay probe to cd and writes {nseg, seg_chunks, lead} to
// plan (device), which the segment pass, the scan and the correction pass
// read; their grids are sized for nseg_max segments.
cudaError_t launch_segment_plan(const float* probe, int nprobe, long long BH, int T, int nsm,
                                int nseg_max, int* plan, cudaStream_t stream);
cudaError_t launch_chunk_fwd_tc_segmented_planned(const ChunkFwdArgs& a, int nseg_max,
                                                  float* ws, const int* plan);

cudaError_t launch_decode(const DecodeArgs& a, kda_dtype_t io);
cudaError_t launch_decode_multi(const MultiDecodeArgs& a, kda_dtype_t io);
cudaError_t launch_selftest_wait(long long limit, int* d_status, cudaStream_t stream);

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------

// Lower log-decay bound (section "A lower bound that deleted a GPU code path"
// of the orkas.ai page "Kimi K3 architecture": at least 0.67% ~ e^-5 of the
// state survives one step).
constexpr float kLogDecayMin = -5.0f;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Programmatic dependent launch: a kernel launched by launch_dependent may
// start while the stream's previous kernel finishes; it calls pdl_wait()
// before reading anything, which returns once that kernel is done (and at
// once for an ordinary launch).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Status bits for one log-decay value: range [-5, 0] and finiteness.
__device__ __forceinline__ int decay_flags(float gv) {
    int f = 0;
    if (!(fabsf(gv) <= 3.402823466e38f)) f |= KDA_DEV_NONFINITE;  // NaN or Inf
    else if (gv < kLogDecayMin || gv > 0.0f) f |= KDA_DEV_DECAY_RANGE;
    return f;
}
__device__ __forceinline__ int finite_flag(float x) {
    return (fabsf(x) <= 3.402823466e38f) ? 0 : KDA_DEV_NONFINITE;
}

// OR a per-thread flag word into *d_status with one atomic per warp.
__device__ __forceinline__ void report_flags(int* d_status, int flags) {
    unsigned m = __activemask();
    int any = __reduce_or_sync(m, flags);
    if (any && d_status && (threadIdx.x & 31) == (__ffs(m) - 1)) atomicOr(d_status, any);
}

}  // namespace kda
