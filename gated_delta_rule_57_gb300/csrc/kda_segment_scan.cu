// Prefix scan over the segments of a sequence split in time.
//
// The recurrence S_t = (I - b k k^T) Diag(e^g) S_{t-1} + b k v^T is affine in
// the state, so a segment maps its incoming state X to M X + S0, where M is
// the product of its per-token transitions (the segment run from the identity
// with v = 0) and S0 its final state from a zero start. The orkas.ai page
// "Kimi K3 architecture" (section "The bill arrives in the serving stack",
// first bullet) splits one long sequence across devices with these two
// composable summaries and a prefix scan over them; here the segments share
// one GPU. Given S0 and M of every segment (the first segment
// starts from h0, so its S0 already is its true final state):
//     X_1 = S0_0,   X_{s+1} = S0_s + M_s X_s   (s = 1 .. nseg - 1),
// X_s is the true incoming state of segment s (written to sin[s - 1]) and
// X_nseg the sequence's final state (written to hT when it is not null).
// Column block c of X_{s+1} depends only on column block c of X_s, so each
// sequence runs on kColBlocks CTAs, one per 32 value columns, with no
// exchange between them; a CTA prefetches the next segment's M and its block
// of S0 (cp.async, two buffers) while it multiplies the current ones. fp32
// throughout; every output element starts from S0 and adds M[i][kk] X[kk][j]
// for kk = 0, 1, .., dk - 1 in that order, whatever the blocking. A transition
// that is exactly zero (a segment whose decay empties any state: its run
// stopped at a zero state) with a finite X adds only zeros, so that step
// keeps X_{s+1} = S0_s without the product (equal values; only the sign of a
// zero entry may differ from adding the zero products); a NaN or Inf in M or
// X takes the product, so it propagates as before.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kDs = 128;                   // dk = dv
constexpr int kCols = 32;                  // value columns per CTA
constexpr int kColBlocks = kDs / kCols;    // CTAs per sequence
constexpr int kLdm = kDs + 4;              // padded M row: the four rows a warp reads hit distinct banks
constexpr int kScanThreads = 128;          // thread: rows i0 + 16 a (a < 8) x columns j0 .. j0 + 3
constexpr int kMFloats = kDs * kLdm;
constexpr int kBFloats = kDs * kCols;
constexpr size_t kScanSmem = (2 * (size_t)kMFloats + 3 * (size_t)kBFloats) * sizeof(float);

// Entry s of sequence bh sits at s0 + (s * s_seg + bh * s_bh) * DD, and
// likewise for m and sin with their own strides (m and sin start at segment 1):
// segment-major within a sequence (the time-segmented prefill) or sequence-
// major within a segment (summaries gathered from the ranks of a sequence
// split across devices).
struct ScanLayout {
    long long s0_seg, s0_bh, m_seg, m_bh, in_seg, in_bh;
};

__device__ __forceinline__ void cp_async16(float* dst, const float* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     (unsigned)__cvta_generic_to_shared(dst)),
                 "l"(__cvta_generic_to_global(src))
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// plan (device, nullable): a device-planned split, whose segment count
// replaces nseg (segment-major layout).
__global__ void __launch_bounds__(kScanThreads, 1)
    kda_segment_scan_kernel(const float* __restrict__ s0, const float* __restrict__ m,
                            float* __restrict__ sin, float* __restrict__ hT, int nseg,
                            ScanLayout L, const int* __restrict__ plan) {
    // Scans of a time split run as programmatic dependents of the segment
    // pass: nothing is read before it is done (a no-op for other launches).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (plan) {  // nseg is the largest plan the workspace holds
        nseg = min(max(__ldg(plan), 1), nseg);
        L = ScanLayout{1, nseg, 1, nseg - 1, 1, nseg - 1};
    }
    extern __shared__ __align__(16) float smem[];
    float* Mb = smem;                      // [2][kDs][kLdm]   M of the current and next segment
    float* Sb = smem + 2 * kMFloats;       // [2][kDs][kCols]  their blocks of S0
    float* X = Sb + 2 * kBFloats;          // [kDs][kCols]     the running incoming state
    const int tid = threadIdx.x;
    const size_t bh = blockIdx.x;
    const int c0 = blockIdx.y * kCols;
    constexpr size_t DD = (size_t)kDs * kDs;
    const int i0 = tid >> 3, j0 = (tid & 7) * 4;

    auto s0_at = [&](int s) { return s0 + ((long long)s * L.s0_seg + (long long)bh * L.s0_bh) * DD; };
    auto m_at = [&](int s) { return m + ((long long)(s - 1) * L.m_seg + (long long)bh * L.m_bh) * DD; };
    auto in_at = [&](int s) { return sin + ((long long)(s - 1) * L.in_seg + (long long)bh * L.in_bh) * DD; };
    // Requests M_s and this CTA's block of S0_s into buffer b, as one group.
    auto stage = [&](int s, int b) {
        const float* ms = m_at(s);
        float* md = Mb + b * kMFloats;
        for (int e = tid; e < kDs * kDs / 4; e += kScanThreads) {
            const int r = e >> 5, c4 = e & 31;
            cp_async16(md + r * kLdm + 4 * c4, ms + (size_t)r * kDs + 4 * c4);
        }
        const float* ss = s0_at(s) + c0;
        float* sd = Sb + b * kBFloats;
        for (int e = tid; e < kBFloats / 4; e += kScanThreads) {
            const int r = e >> 3, c4 = e & 7;
            cp_async16(sd + r * kCols + 4 * c4, ss + (size_t)r * kDs + 4 * c4);
        }
        cp_async_commit();
    };

    if (nseg > 1) stage(1, 0);
    // X_1 = S0_0: the incoming state of segment 1 (entry 0 of sin), or hT
    {
        const float* src = s0_at(0) + c0;
        float* copy_to = nseg > 1 ? in_at(1) + c0 : (hT ? hT + bh * DD + c0 : nullptr);
        for (int e = tid; e < kBFloats / 4; e += kScanThreads) {
            const int r = e >> 3, c4 = e & 7;
            const float4 f = *reinterpret_cast<const float4*>(src + (size_t)r * kDs + 4 * c4);
            *reinterpret_cast<float4*>(X + r * kCols + 4 * c4) = f;
            if (copy_to) *reinterpret_cast<float4*>(copy_to + (size_t)r * kDs + 4 * c4) = f;
        }
    }
    for (int s = 1; s < nseg; s++) {
        const int b = (s - 1) & 1;
        if (s + 1 < nseg) {
            stage(s + 1, b ^ 1);  // its buffer was last read before the previous step's barrier
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();  // M_s, S0_s and X visible to every thread
        const float* Ms = Mb + b * kMFloats;
        const float* Ss = Sb + b * kBFloats;
        bool need = false;  // a nonzero (or NaN) entry of M_s, or a non-finite one of X
        for (int e = tid; e < kDs * kDs / 4; e += kScanThreads) {
            const float4 f = *reinterpret_cast<const float4*>(Ms + (e >> 5) * kLdm + 4 * (e & 31));
            need = need || f.x != 0.f || f.y != 0.f || f.z != 0.f || f.w != 0.f;
        }
        for (int e = tid; e < kBFloats / 4; e += kScanThreads) {
            const float4 f = *reinterpret_cast<const float4*>(X + 4 * e);
            need = need || !isfinite(f.x) || !isfinite(f.y) || !isfinite(f.z) || !isfinite(f.w);
        }
        need = __syncthreads_or(need);
        float acc[8][4];
#pragma unroll
        for (int a = 0; a < 8; a++) {
            const float4 f = *reinterpret_cast<const float4*>(Ss + (i0 + 16 * a) * kCols + j0);
            acc[a][0] = f.x; acc[a][1] = f.y; acc[a][2] = f.z; acc[a][3] = f.w;
        }
        if (need) {
#pragma unroll 2
            for (int kk = 0; kk < kDs; kk += 4) {
                float4 mv[8], xv[4];
#pragma unroll
                for (int a = 0; a < 8; a++)
                    mv[a] = *reinterpret_cast<const float4*>(Ms + (i0 + 16 * a) * kLdm + kk);
#pragma unroll
                for (int q = 0; q < 4; q++)
                    xv[q] = *reinterpret_cast<const float4*>(X + (kk + q) * kCols + j0);
#pragma unroll
                for (int a = 0; a < 8; a++) {
                    const float mm[4] = {mv[a].x, mv[a].y, mv[a].z, mv[a].w};
#pragma unroll
                    for (int q = 0; q < 4; q++) {
                        acc[a][0] = fmaf(mm[q], xv[q].x, acc[a][0]);
                        acc[a][1] = fmaf(mm[q], xv[q].y, acc[a][1]);
                        acc[a][2] = fmaf(mm[q], xv[q].z, acc[a][2]);
                        acc[a][3] = fmaf(mm[q], xv[q].w, acc[a][3]);
                    }
                }
            }
        }
        __syncthreads();  // every thread is done reading X and buffer b
        float* out = s + 1 < nseg ? in_at(s + 1) : (hT ? hT + bh * DD : nullptr);
#pragma unroll
        for (int a = 0; a < 8; a++) {
            const int r = i0 + 16 * a;
            const float4 f = make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
            *reinterpret_cast<float4*>(X + r * kCols + j0) = f;
            if (out) *reinterpret_cast<float4*>(out + (size_t)r * kDs + c0 + j0) = f;
        }
    }
}

}  // namespace

// dependent: launched as a programmatic dependent of the stream's previous
// kernel (the scan waits for it before reading anything).
static cudaError_t launch_scan(const float* s0, const float* m, float* sin, float* hT, int BH,
                               int nseg, const ScanLayout& L, cudaStream_t stream,
                               const int* plan = nullptr, bool dependent = false) {
    cudaError_t e = cudaFuncSetAttribute(kda_segment_scan_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kScanSmem);
    if (e != cudaSuccess) return e;
    if (!dependent) {
        kda_segment_scan_kernel<<<dim3(BH, kColBlocks), kScanThreads, kScanSmem, stream>>>(
            s0, m, sin, hT, nseg, L, plan);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(BH, kColBlocks);
    cfg.blockDim = dim3(kScanThreads);
    cfg.dynamicSmemBytes = kScanSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kda_segment_scan_kernel, s0, m, sin, hT, nseg, L, plan);
}

cudaError_t launch_segment_scan(const float* s0, const float* m, float* sin, float* hT, int BH,
                                int nseg, cudaStream_t stream) {
    const ScanLayout L{1, nseg, 1, nseg - 1, 1, nseg - 1};
    return launch_scan(s0, m, sin, hT, BH, nseg, L, stream, nullptr, true);
}

cudaError_t launch_segment_scan_planned(const float* s0, const float* m, float* sin, float* hT,
                                        int BH, int nseg_max, const int* plan,
                                        cudaStream_t stream) {
    const ScanLayout L{1, 1, 1, 1, 1, 1};  // replaced from the plan in the kernel
    return launch_scan(s0, m, sin, hT, BH, nseg_max, L, stream, plan, true);
}

cudaError_t launch_slice_scan(const float* s0, const float* m, float* sin, float* hT, int BH,
                              int nslice, cudaStream_t stream) {
    const ScanLayout L{BH, 1, BH, 1, BH, 1};
    return launch_scan(s0, m, sin, hT, BH, nslice, L, stream);
}

}  // namespace kda
