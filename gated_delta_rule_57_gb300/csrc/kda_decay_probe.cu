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
// the plan only: results never depend on it. A CTA takes one sample of one
// batch row for hpc heads (2, so that a few heads still spread over the SMs;
// 8 when H needs it to fit the grid); four warps per head read 16 of the
// chunk's rows each (dk contiguous floats per row), all loads in flight before
// any is used, and the four partial sums are added in token order.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kProbeHeads = 8;   // most heads per CTA
constexpr int kProbeParts = 4;   // warps per head, 16 tokens each
constexpr int kProbeRows = 16;   // rows of g in flight per warp

template <int DK>
__global__ void __launch_bounds__(32 * kProbeHeads * kProbeParts)
    kda_decay_probe_kernel(const float* __restrict__ g, int T, int H, int nsample, int hpc,
                           float* __restrict__ out) {
    constexpr int PER = DK / 32;  // floats per lane of a row: 4 or 2
    __shared__ float s_part[kProbeHeads][kProbeParts];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hl = warp / kProbeParts, part = warp % kProbeParts;
    const int s = blockIdx.x, b = blockIdx.y, h = blockIdx.z * hpc + hl;
    const int nch = (T + 63) / 64;
    const int c = (int)(((long long)s * nch) / nsample);
    const int t0 = c * 64 + part * kProbeRows, t1 = min(T, c * 64 + 64);
    float sum = 0.f;
    if (h < H && t0 < t1) {
        const float* base = g + (((size_t)b * T) * H + h) * DK + PER * lane;
        const size_t row_stride = (size_t)H * DK;  // next token, same head
        float m[kProbeRows];
        if (t0 + kProbeRows <= t1) {  // a whole group: every load out before any use
            if constexpr (PER == 4) {
                float4 f[kProbeRows];
#pragma unroll
                for (int u = 0; u < kProbeRows; u++)
                    f[u] = __ldcs(reinterpret_cast<const float4*>(base + (size_t)(t0 + u) * row_stride));
#pragma unroll
                for (int u = 0; u < kProbeRows; u++)
                    m[u] = fmaxf(fmaxf(f[u].x, f[u].y), fmaxf(f[u].z, f[u].w));
            } else {
                float2 f[kProbeRows];
#pragma unroll
                for (int u = 0; u < kProbeRows; u++)
                    f[u] = __ldcs(reinterpret_cast<const float2*>(base + (size_t)(t0 + u) * row_stride));
#pragma unroll
                for (int u = 0; u < kProbeRows; u++) m[u] = fmaxf(f[u].x, f[u].y);
            }
        } else {  // the short last chunk
#pragma unroll
            for (int u = 0; u < kProbeRows; u++) {
                m[u] = -INFINITY;
                if (t0 + u < t1) {
                    const float* r = base + (size_t)(t0 + u) * row_stride;
                    m[u] = r[0];
#pragma unroll
                    for (int e = 1; e < PER; e++) m[u] = fmaxf(m[u], r[e]);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kProbeRows; u++) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                m[u] = fmaxf(m[u], __shfl_xor_sync(0xffffffffu, m[u], off));
        }
#pragma unroll
        for (int u = 0; u < kProbeRows; u++)
            if (t0 + u < t1) sum += m[u];
    }
    if (lane == 0) s_part[hl][part] = sum;
    __syncthreads();
    if ((int)threadIdx.x < hpc) {
        const int hh = blockIdx.z * hpc + threadIdx.x;
        if (hh < H) {
            float tot = 0.f;
#pragma unroll
            for (int p = 0; p < kProbeParts; p++) tot += s_part[threadIdx.x][p];  // token order
            out[((size_t)b * nsample + s) * H + hh] = tot;
        }
    }
}

// The split of a device-planned segmented prefill, from a decay probe: the
// largest finite entry is cd (none, or a non-finite one: whole-segment runs,
// as without a probe). Warp w takes the segment counts 2 + w and 18 + w, its
// lanes the first-segment lengths 1 .. 16, and reduces them to the count's
// best (cost, lead); one thread then takes the same choice over the counts as
// the host's kda_chunk_fwd_segments_hint_decay and writes {nseg, seg_chunks,
// lead}. Costs use 32-bit arithmetic when every value fits (the same
// numbers), else 64-bit.
constexpr int kPlanThreads = 512;

__global__ void __launch_bounds__(kPlanThreads)
    kda_segment_plan_kernel(const float* __restrict__ probe, int nprobe, long long BH, int T,
                            int nsm, int nseg_max, int* __restrict__ plan) {
    // Launched as a programmatic dependent of the probe: wait for it first.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    __shared__ float s_max[kPlanThreads / 32];
    __shared__ int s_bad[kPlanThreads / 32];
    __shared__ long long s_bc[kPlanMaxSeg + 1];
    __shared__ int s_bl[kPlanMaxSeg + 1];
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
    const bool fits = plan_fits_32(BH, T, nsm);
    const int l = lane + 1;
    for (int k = 0; k < 2; k++) {
        const int sg = 2 + warp + 16 * k;
        long long c = -1;
        if (sg <= kPlanMaxSeg && l <= kPlanMaxLead && nsm > 0)
            c = fits ? (long long)split_cost_t<int>((int)BH, T, sg, l, nsm, (int)tl)
                     : split_cost(BH, T, sg, l, nsm, tl);
        // lead 1 decides whether the count is usable; then the least cost,
        // the smallest lead among equal ones
        const long long c1 = __shfl_sync(0xffffffffu, c, 0);
        long long bc = c >= 0 ? c : 0x7fffffffffffffffLL;
        int bl = l;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const long long oc = __shfl_xor_sync(0xffffffffu, bc, off);
            const int ol = __shfl_xor_sync(0xffffffffu, bl, off);
            if (oc < bc || (oc == bc && ol < bl)) {
                bc = oc;
                bl = ol;
            }
        }
        if (lane == 0 && sg <= kPlanMaxSeg) {
            s_bc[sg] = c1 < 0 ? c1 : bc;
            s_bl[sg] = c1 < 0 ? 1 : bl;
        }
    }
    __syncthreads();
    if (tid == 0) {
        const SegPlan sp = choose_plan_best(BH, T, nsm, nseg_max, s_bc, s_bl);
        plan[0] = sp.nseg;
        plan[1] = sp.seg_chunks;
        plan[2] = sp.lead;
    }
}

}  // namespace

cudaError_t launch_decay_probe(const float* g, int B, int T, int H, int dk, int nsample,
                               float* out, cudaStream_t stream) {
    const int hpc = (H + 1) / 2 <= 65535 ? 2 : kProbeHeads;
    const dim3 grid((unsigned)nsample, (unsigned)B, (unsigned)((H + hpc - 1) / hpc));
    const int threads = 32 * hpc * kProbeParts;
    if (dk == 128)
        kda_decay_probe_kernel<128><<<grid, threads, 0, stream>>>(g, T, H, nsample, hpc, out);
    else
        kda_decay_probe_kernel<64><<<grid, threads, 0, stream>>>(g, T, H, nsample, hpc, out);
    return cudaGetLastError();
}

cudaError_t launch_segment_plan(const float* probe, int nprobe, long long BH, int T, int nsm,
                                int nseg_max, int* plan, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(kPlanThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kda_segment_plan_kernel, probe, nprobe, BH, T, nsm, nseg_max,
                              plan);
}

}  // namespace kda
