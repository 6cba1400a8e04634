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
