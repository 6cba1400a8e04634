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
// fp32 throughout; one CTA per sequence, the running X and the current M in
// shared memory.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kDs = 128;       // dk = dv
constexpr int kLd = kDs + 4;   // padded row: column reads of M fall on distinct banks
constexpr int kScanThreads = 256;
constexpr size_t kScanSmem = 2 * (size_t)kDs * kLd * sizeof(float);

// Entry s of sequence bh sits at s0 + (s * s_seg + bh * s_bh) * DD, and
// likewise for m and sin with their own strides (m and sin start at segment 1):
// segment-major within a sequence (the time-segmented prefill) or sequence-
// major within a segment (summaries gathered from the ranks of a sequence
// split across devices).
struct ScanLayout {
    long long s0_seg, s0_bh, m_seg, m_bh, in_seg, in_bh;
};

__global__ void __launch_bounds__(kScanThreads)
    kda_segment_scan_kernel(const float* __restrict__ s0, const float* __restrict__ m,
                            float* __restrict__ sin, float* __restrict__ hT, int nseg,
                            const ScanLayout L) {
    extern __shared__ __align__(16) float smem[];
    float* X = smem;              // [kDs][kLd]
    float* Ms = smem + kDs * kLd;  // [kDs][kLd]
    const int tid = threadIdx.x;
    const size_t bh = blockIdx.x;
    constexpr size_t DD = (size_t)kDs * kDs;
    const int i0 = (tid >> 4) * 8, j0 = (tid & 15) * 8;  // this thread's 8 x 8 output tile

    // Copies a dk x dv state into a padded shared-memory tile (and to copy_to).
    auto load = [&](float* dst, const float* src, float* copy_to) {
        for (int e = tid; e < kDs * kDs / 4; e += kScanThreads) {
            const int r = e / (kDs / 4), c4 = e % (kDs / 4);
            const float4 f = *reinterpret_cast<const float4*>(src + (size_t)r * kDs + 4 * c4);
            *reinterpret_cast<float4*>(dst + r * kLd + 4 * c4) = f;
            if (copy_to) *reinterpret_cast<float4*>(copy_to + (size_t)r * kDs + 4 * c4) = f;
        }
    };
    auto s0_at = [&](int s) { return s0 + ((long long)s * L.s0_seg + (long long)bh * L.s0_bh) * DD; };
    auto m_at = [&](int s) { return m + ((long long)(s - 1) * L.m_seg + (long long)bh * L.m_bh) * DD; };
    auto in_at = [&](int s) { return sin + ((long long)(s - 1) * L.in_seg + (long long)bh * L.in_bh) * DD; };
    // X_1 = S0_0, the incoming state of segment 1 (entry 0 of sin)
    load(X, s0_at(0), nseg > 1 ? in_at(1) : nullptr);
    if (nseg == 1 && hT) load(X, s0_at(0), hT + bh * DD);
    for (int s = 1; s < nseg; s++) {
        load(Ms, m_at(s), nullptr);
        __syncthreads();
        float acc[8][8];
        const float* s0s = s0_at(s);
#pragma unroll
        for (int a = 0; a < 8; a++) {
#pragma unroll
            for (int c = 0; c < 8; c += 4) {
                const float4 f = *reinterpret_cast<const float4*>(s0s + (size_t)(i0 + a) * kDs + j0 + c);
                acc[a][c] = f.x; acc[a][c + 1] = f.y; acc[a][c + 2] = f.z; acc[a][c + 3] = f.w;
            }
        }
        for (int kk = 0; kk < kDs; kk++) {
            float mv[8], xv[8];
#pragma unroll
            for (int a = 0; a < 8; a++) mv[a] = Ms[(i0 + a) * kLd + kk];
            const float4 x0 = *reinterpret_cast<const float4*>(X + kk * kLd + j0);
            const float4 x1 = *reinterpret_cast<const float4*>(X + kk * kLd + j0 + 4);
            xv[0] = x0.x; xv[1] = x0.y; xv[2] = x0.z; xv[3] = x0.w;
            xv[4] = x1.x; xv[5] = x1.y; xv[6] = x1.z; xv[7] = x1.w;
#pragma unroll
            for (int a = 0; a < 8; a++) {
#pragma unroll
                for (int c = 0; c < 8; c++) acc[a][c] = fmaf(mv[a], xv[c], acc[a][c]);
            }
        }
        __syncthreads();  // every thread is done reading X and M
        float* out = s + 1 < nseg ? in_at(s + 1) : (hT ? hT + bh * DD : nullptr);
#pragma unroll
        for (int a = 0; a < 8; a++) {
#pragma unroll
            for (int c = 0; c < 8; c += 4) {
                const float4 f = make_float4(acc[a][c], acc[a][c + 1], acc[a][c + 2], acc[a][c + 3]);
                *reinterpret_cast<float4*>(X + (i0 + a) * kLd + j0 + c) = f;
                if (out) *reinterpret_cast<float4*>(out + (size_t)(i0 + a) * kDs + j0 + c) = f;
            }
        }
        __syncthreads();
    }
}

}  // namespace

static cudaError_t launch_scan(const float* s0, const float* m, float* sin, float* hT, int BH,
                               int nseg, const ScanLayout& L, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(kda_segment_scan_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kScanSmem);
    if (e != cudaSuccess) return e;
    kda_segment_scan_kernel<<<BH, kScanThreads, kScanSmem, stream>>>(s0, m, sin, hT, nseg, L);
    return cudaGetLastError();
}

cudaError_t launch_segment_scan(const float* s0, const float* m, float* sin, float* hT, int BH,
                                int nseg, cudaStream_t stream) {
    const ScanLayout L{1, nseg, 1, nseg - 1, 1, nseg - 1};
    return launch_scan(s0, m, sin, hT, BH, nseg, L, stream);
}

cudaError_t launch_slice_scan(const float* s0, const float* m, float* sin, float* hT, int BH,
                              int nslice, cudaStream_t stream) {
    const ScanLayout L{BH, 1, BH, 1, BH, 1};
    return launch_scan(s0, m, sin, hT, BH, nslice, L, stream);
}

}  // namespace kda
