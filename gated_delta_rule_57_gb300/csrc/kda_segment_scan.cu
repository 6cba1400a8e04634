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

__global__ void __launch_bounds__(kScanThreads)
    kda_segment_scan_kernel(const float* __restrict__ s0, const float* __restrict__ m,
                            float* __restrict__ sin, float* __restrict__ hT, int nseg) {
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
    // X_1 = S0_0, the incoming state of segment 1 (entry 0 of sin)
    load(X, s0 + bh * nseg * DD, sin + bh * (nseg - 1) * DD);
    for (int s = 1; s < nseg; s++) {
        load(Ms, m + (bh * (nseg - 1) + s - 1) * DD, nullptr);
        __syncthreads();
        float acc[8][8];
        const float* s0s = s0 + (bh * nseg + s) * DD;
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
        float* out = s + 1 < nseg ? sin + (bh * (nseg - 1) + s) * DD : (hT ? hT + bh * DD : nullptr);
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

cudaError_t launch_segment_scan(const float* s0, const float* m, float* sin, float* hT, int BH,
                                int nseg, cudaStream_t stream) {
    cudaError_t e = cudaFuncSetAttribute(kda_segment_scan_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kScanSmem);
    if (e != cudaSuccess) return e;
    kda_segment_scan_kernel<<<BH, kScanThreads, kScanSmem, stream>>>(s0, m, sin, hT, nseg);
    return cudaGetLastError();
}

}  // namespace kda
