// Sampled bound on how fast the decay empties a state, for planning a
// sequence split in time.
//
// In the recurrence S_t = (I - b_t k_t k_t^T) Diag(e^{g_t}) S_{t-1} + b_t k_t v_t^T
// (the orkas.ai page "Kimi K3 architecture"), a run with v = 0 (a segment's
// transition from the identity, or a correction from a segment's incoming
// state) only multiplies its state by (I - b k k^T) Diag(e^g). For a unit key
// and 0 <= b <= 2 the first factor is a contraction, so over one 64-token chunk
// the state's largest entry shrinks at least by e^{sum_t max_c g_t,c}. Once
// that product has passed fp32's smallest subnormal (2^-149 ~ e^-103.3) the
// state is exactly zero and such a run stops (the segmented prefill checks for
// it after every chunk). This kernel evaluates sum_t max_c g over a sample of
// chunks: entry [b][s][h] is that sum for head h over the tokens of chunk
// floor(s * nch / nsample) of batch row b (a short last chunk sums its tokens
// only). The planner takes the largest entry as the decay per chunk that the
// sequences can be counted on; it is an estimate from a sample, so it guides
// the plan only: results never depend on it. One warp per (sample, row,
// head) reads the chunk's rows of that head (dk contiguous floats each) 16 at
// a time, so that many loads are in flight per lane.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kProbeWarps = 8;
constexpr int kProbeRows = 16;  // rows of g in flight per warp

template <int DK>
__global__ void __launch_bounds__(32 * kProbeWarps)
    kda_decay_probe_kernel(const float* __restrict__ g, int T, int H, int nsample,
                           float* __restrict__ out) {
    constexpr int PER = DK / 32;  // floats per lane of a row: 4 or 2
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int s = blockIdx.x, b = blockIdx.y, h = blockIdx.z * kProbeWarps + warp;
    if (h >= H) return;
    const int nch = (T + 63) / 64;
    const int c = (int)(((long long)s * nch) / nsample);
    const int t0 = c * 64, t1 = min(T, t0 + 64);
    const float* base = g + (((size_t)b * T) * H + h) * DK + PER * lane;
    const size_t row_stride = (size_t)H * DK;  // next token, same head
    float sum = 0.f;
    if (t1 - t0 == 64) {  // a whole chunk: the loads of a group go out before any is used
        for (int t = t0; t < t1; t += kProbeRows) {
            float m[kProbeRows];
            if constexpr (PER == 4) {
                float4 f[kProbeRows];
#pragma unroll
                for (int u = 0; u < kProbeRows; u++)
                    f[u] = __ldcs(reinterpret_cast<const float4*>(base + (size_t)(t + u) * row_stride));
#pragma unroll
                for (int u = 0; u < kProbeRows; u++)
                    m[u] = fmaxf(fmaxf(f[u].x, f[u].y), fmaxf(f[u].z, f[u].w));
            } else {
                float2 f[kProbeRows];
#pragma unroll
                for (int u = 0; u < kProbeRows; u++)
                    f[u] = __ldcs(reinterpret_cast<const float2*>(base + (size_t)(t + u) * row_stride));
#pragma unroll
                for (int u = 0; u < kProbeRows; u++) m[u] = fmaxf(f[u].x, f[u].y);
            }
#pragma unroll
            for (int u = 0; u < kProbeRows; u++) {
#pragma unroll
                for (int off = 16; off > 0; off >>= 1)
                    m[u] = fmaxf(m[u], __shfl_xor_sync(0xffffffffu, m[u], off));
            }
#pragma unroll
            for (int u = 0; u < kProbeRows; u++) sum += m[u];
        }
    } else {  // the short last chunk
        for (int t = t0; t < t1; t++) {
            const float* r = base + (size_t)t * row_stride;
            float m = r[0];
#pragma unroll
            for (int e = 1; e < PER; e++) m = fmaxf(m, r[e]);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
            sum += m;
        }
    }
    if (lane == 0) out[((size_t)b * nsample + s) * H + h] = sum;
}

// The split of a device-planned segmented prefill, from a decay probe: the
// largest finite entry is cd (none, or a non-finite one: whole-segment runs,
// as without a probe); the threads fill the cost table of every (segment
// count, first-segment length), and one thread takes the same choice as the
// host's kda_chunk_fwd_segments_hint_decay, writing {nseg, seg_chunks, lead}.
constexpr int kPlanThreads = 512;

__global__ void __launch_bounds__(kPlanThreads)
    kda_segment_plan_kernel(const float* __restrict__ probe, int nprobe, long long BH, int T,
                            int nsm, int nseg_max, int* __restrict__ plan) {
    __shared__ float s_max[kPlanThreads / 32];
    __shared__ int s_bad[kPlanThreads / 32];
    __shared__ long long s_cost[kPlanCosts];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float m = -INFINITY;
    int bad = 0;
    for (int i = tid; i < nprobe; i += kPlanThreads) {
        const float x = probe[i];
        if (isfinite(x)) m = fmaxf(m, x);
        else bad = 1;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        bad |= __shfl_xor_sync(0xffffffffu, bad, off);
    }
    if (lane == 0) {
        s_max[warp] = m;
        s_bad[warp] = bad;
    }
    __syncthreads();
    float cd = -INFINITY;
    int any_bad = 0;
    for (int w = 0; w < kPlanThreads / 32; w++) {
        cd = fmaxf(cd, s_max[w]);
        any_bad |= s_bad[w];
    }
    if (nprobe == 0 || any_bad) cd = 0.f;
    const long long tl = transition_chunks(cd, T);
    for (int e = tid; e < kPlanCosts; e += kPlanThreads) {
        const int sg = e / kPlanStride, l = e % kPlanStride;
        s_cost[e] = (sg >= 2 && l >= 1 && nsm > 0) ? split_cost(BH, T, sg, l, nsm, tl) : -1;
    }
    __syncthreads();
    if (tid == 0) {
        const SegPlan sp = choose_plan(BH, T, nsm, nseg_max, s_cost);
        plan[0] = sp.nseg;
        plan[1] = sp.seg_chunks;
        plan[2] = sp.lead;
    }
}

}  // namespace

cudaError_t launch_decay_probe(const float* g, int B, int T, int H, int dk, int nsample,
                               float* out, cudaStream_t stream) {
    const dim3 grid((unsigned)nsample, (unsigned)B, (unsigned)((H + kProbeWarps - 1) / kProbeWarps));
    if (dk == 128)
        kda_decay_probe_kernel<128><<<grid, 32 * kProbeWarps, 0, stream>>>(g, T, H, nsample, out);
    else
        kda_decay_probe_kernel<64><<<grid, 32 * kProbeWarps, 0, stream>>>(g, T, H, nsample, out);
    return cudaGetLastError();
}

cudaError_t launch_segment_plan(const float* probe, int nprobe, long long BH, int T, int nsm,
                                int nseg_max, int* plan, cudaStream_t stream) {
    kda_segment_plan_kernel<<<1, kPlanThreads, 0, stream>>>(probe, nprobe, BH, T, nsm, nseg_max,
                                                            plan);
    return cudaGetLastError();
}

}  // namespace kda
