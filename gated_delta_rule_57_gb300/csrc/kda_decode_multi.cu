// KDA multi-token decode: K cached tokens per sequence applied to the fp32
// state in one pass (speculative decoding).
//
// The orkas.ai page "Kimi K3 architecture" (section "The bill arrives in the
// serving stack", third bullet) notes that the state is updated in place, so a
// rejected draft cannot be undone by restoring an older state; instead the
// projected inputs of the draft tokens (far smaller than the state) are cached
// and the state is rebuilt on chip. This kernel serves both halves:
//   verify (commit = 0): outputs o_t for all K draft tokens, state untouched;
//   commit (commit = 1): the state advanced by the accepted prefix ntok[n] of
//                        each sequence, written back in place (o optional).
// Per token it is the decode recurrence
//     S' = Diag(exp g) S,  u = beta (v - S'^T k),  S = S' + k u^T,
//     o  = S^T q = S'^T q + u (k . q).
// The state slice stays in registers for all K tokens: it is read once and
// written at most once, so K tokens cost about the HBM traffic of one
// single-token step.
#include "kda_internal.cuh"

namespace kda {
namespace {

// One CTA per (sequence, head, DVS-wide slice of the value columns): the
// columns of S evolve independently given k, g, beta, so a slice only needs
// its own v columns. Small CTAs let several per SM overlap one CTA's per-token
// reductions with another's state streaming.
template <typename TIn, int DK, int DVS, int NT>
__global__ void __launch_bounds__(NT, 512 / NT)
    kda_decode_multi_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k,
                            const TIn* __restrict__ v, const float* __restrict__ g,
                            const float* __restrict__ beta, float* __restrict__ S,
                            TIn* __restrict__ o, const int* __restrict__ ntok, int K, int H,
                            int DV, int commit, int* __restrict__ d_status) {
    constexpr int CG = DVS / 4;   // float4 column groups per state row slice
    constexpr int RG = NT / CG;   // row groups
    constexpr int RPT = DK / RG;  // rows per thread
    constexpr int NW = NT / 32;
    static_assert(NT % CG == 0 && DK % RG == 0, "bad tiling");

    // Token vectors and reduction buffers are double-buffered by token parity,
    // so a token costs three barriers.
    __shared__ float s_k[2][DK], s_q[2][DK], s_a[2][DK];
    __shared__ float s_red[2][2][RG][DVS];
    __shared__ __align__(16) float s_tot[2][2][DVS];  // column totals of S'^T k and S'^T q
    static_assert(NT == 2 * DVS, "one thread per (column, reduction)");
    __shared__ float s_kq[2][NW];

    const int tid = threadIdx.x;
    const size_t head = blockIdx.x;  // n * H + h
    const int n = (int)(head / H), hh = (int)(head % H);
    const int j0 = blockIdx.y * DVS;  // first value column of this slice
    const int cg = tid % CG, rg = tid / CG;
    const int RS = DV / 4;  // float4 per full state row
    int nt = K;
    if (ntok) nt = min(max(ntok[n], 0), K);
    float4* Sh = reinterpret_cast<float4*>(S + head * DK * DV + j0);

    float4 st[RPT];
#pragma unroll
    for (int r = 0; r < RPT; r++) st[r] = Sh[(size_t)(rg + r * RG) * RS + cg];

    // The next token's inputs are loaded into registers while the current one
    // is processed, so their HBM latency is off the per-token chain.
    constexpr int PER = (DK + NT - 1) / NT;  // key channels per thread (<= 1 here)
    float nk[PER], nq[PER], ng[PER], nv[4], nb = 0.f;
    auto fetch = [&](int t) {
        const size_t row = ((size_t)n * K + t) * H + hh;
#pragma unroll
        for (int p = 0; p < PER; p++) {
            const int i = tid + p * NT;
            if (i < DK) {
                nk[p] = to_f32(k[row * DK + i]);
                nq[p] = to_f32(q[row * DK + i]);
                ng[p] = g[row * DK + i];
            }
        }
#pragma unroll
        for (int c = 0; c < 4; c++) nv[c] = to_f32(v[row * DV + j0 + cg * 4 + c]);
        nb = beta[row];
    };
    if (nt > 0) fetch(0);

    int flags = 0;
    for (int t = 0; t < nt; t++) {
        const int buf = t & 1;
        const size_t row = ((size_t)n * K + t) * H + hh;
        float kq = 0.f;
#pragma unroll
        for (int p = 0; p < PER; p++) {
            const int i = tid + p * NT;
            if (i < DK) {
                flags |= decay_flags(ng[p]);
                s_k[buf][i] = nk[p];
                s_q[buf][i] = nq[p];
                s_a[buf][i] = expf(ng[p]);
                kq += nk[p] * nq[p];
            }
        }
        const float b = nb;
        float vj[4];
#pragma unroll
        for (int c = 0; c < 4; c++) vj[c] = nv[c];
        if (tid == 0) flags |= finite_flag(b);
        if (t + 1 < nt) fetch(t + 1);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
        if ((tid & 31) == 0) s_kq[buf][tid >> 5] = kq;
        __syncthreads();

        float pk[4] = {0.f, 0.f, 0.f, 0.f}, pq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int r = 0; r < RPT; r++) {
            const int i = rg + r * RG;
            const float a = s_a[buf][i], ki = s_k[buf][i], qi = s_q[buf][i];
            st[r].x *= a;
            st[r].y *= a;
            st[r].z *= a;
            st[r].w *= a;
            pk[0] += st[r].x * ki;
            pk[1] += st[r].y * ki;
            pk[2] += st[r].z * ki;
            pk[3] += st[r].w * ki;
            pq[0] += st[r].x * qi;
            pq[1] += st[r].y * qi;
            pq[2] += st[r].z * qi;
            pq[3] += st[r].w * qi;
        }
#pragma unroll
        for (int c = 0; c < 4; c++) {
            s_red[buf][0][rg][cg * 4 + c] = pk[c];
            s_red[buf][1][rg][cg * 4 + c] = pq[c];
        }
        __syncthreads();

        {  // thread tid sums one column total over the RG row groups
            const int which = tid / DVS, col = tid % DVS;
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < RG; w++) acc += s_red[buf][which][w][col];
            s_tot[buf][which][col] = acc;
        }
        __syncthreads();
        float kqt = 0.f;
#pragma unroll
        for (int w = 0; w < NW; w++) kqt += s_kq[buf][w];
        float u[4];
        const float4 kv4 = *reinterpret_cast<const float4*>(&s_tot[buf][0][cg * 4]);
        const float4 qv4 = *reinterpret_cast<const float4*>(&s_tot[buf][1][cg * 4]);
        const float kvs[4] = {kv4.x, kv4.y, kv4.z, kv4.w};
        const float qvs[4] = {qv4.x, qv4.y, qv4.z, qv4.w};
#pragma unroll
        for (int c = 0; c < 4; c++) {
            u[c] = b * (vj[c] - kvs[c]);
            if (o && rg == 0) o[row * DV + j0 + cg * 4 + c] = from_f32<TIn>(qvs[c] + u[c] * kqt);
        }
#pragma unroll
        for (int r = 0; r < RPT; r++) {
            const float ki = s_k[buf][rg + r * RG];
            st[r].x += ki * u[0];
            st[r].y += ki * u[1];
            st[r].z += ki * u[2];
            st[r].w += ki * u[3];
        }
    }
    if (commit && nt > 0) {
#pragma unroll
        for (int r = 0; r < RPT; r++) Sh[(size_t)(rg + r * RG) * RS + cg] = st[r];
    }
    report_flags(d_status, flags);
}

template <typename TIn, int D>
cudaError_t launch_t(const MultiDecodeArgs& a) {
    constexpr int DVS = 32, NT = 64;
    const dim3 grid((unsigned)((long long)a.N * a.H), D / DVS);
    kda_decode_multi_kernel<TIn, D, DVS, NT><<<grid, NT, 0, a.stream>>>(
        static_cast<const TIn*>(a.q), static_cast<const TIn*>(a.k),
        static_cast<const TIn*>(a.v), a.g, a.beta, a.S, static_cast<TIn*>(a.o), a.ntok, a.K,
        a.H, D, a.commit, a.d_status);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_multi(const MultiDecodeArgs& a, kda_dtype_t io) {
    if (io == KDA_BF16) return a.dk == 128 ? launch_t<__nv_bfloat16, 128>(a)
                                           : launch_t<__nv_bfloat16, 64>(a);
    return a.dk == 128 ? launch_t<float, 128>(a) : launch_t<float, 64>(a);
}

}  // namespace kda
