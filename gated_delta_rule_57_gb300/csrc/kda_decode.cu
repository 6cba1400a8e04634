// KDA decode step: one token per sequence, fp32 state updated in place.
//
// Per head (the recurrence of the orkas.ai page "Kimi K3 architecture";
// in-place update from section "The bill arrives in the serving stack"):
//     S' = Diag(exp g) S
//     u  = beta (v - S'^T k)
//     S  = S' + k u^T
//     o  = S^T q  =  S'^T q + u (k . q)
// The last identity lets both reductions over the key channel (S'^T k and
// S'^T q) share one pass over S, so S is read once and written once.
//
// Memory plan. Two CTAs per (sequence, head), each owning half of the value
// columns (the columns of S evolve independently given k, g, beta); the two
// halves of a head are adjacent blocks. Each CTA's half of the dk x dv fp32
// state (32 KB at d = 128) is read with 16-byte loads (a warp reads two
// 256-byte row halves), kept in registers across the reduction (16 rows x 4
// columns per thread), and written back in place from the same registers.
// Small CTAs (four per SM) keep one another's loads, arithmetic and stores
// overlapped. The kernel is bound by HBM bandwidth: 2 * dk * dv * 4 bytes of
// state traffic per head against ~5 flops per state element.
#include "kda_internal.cuh"

namespace kda {
namespace {

// DVS: value columns per CTA (a slice of the DV columns of a head; the
// slices of one head are adjacent blocks).
template <typename TIn, int DK, int DV, int DVS, int NT>
__global__ void __launch_bounds__(NT, 512 / NT)
    kda_decode_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k,
                      const TIn* __restrict__ v, const float* __restrict__ g,
                      const float* __restrict__ beta, float* __restrict__ S,
                      TIn* __restrict__ o, int* __restrict__ d_status) {
    constexpr int CG = DVS / 4;        // float4 column groups per row slice
    constexpr int RG = NT / CG;        // row groups (rows handled in parallel)
    constexpr int RPT = DK / RG;       // rows per thread
    constexpr int NW = NT / 32;
    static_assert(NT % CG == 0 && DK % RG == 0, "bad decode tiling");

    __shared__ float s_k[DK], s_q[DK], s_a[DK];
    __shared__ float s_red[2][RG][DVS];
    __shared__ float s_kq[NW];

    pdl_wait();  // the previous step (or whatever came before) is done
    const int tid = threadIdx.x;
    constexpr int NS = DV / DVS;
    const size_t head = blockIdx.x / NS;  // n * H + h
    const int j0 = (int)(blockIdx.x % NS) * DVS;
    const int cg = tid % CG, rg = tid / CG;
    float4* Sh = reinterpret_cast<float4*>(S + head * DK * DV + j0);

    // Issue the state loads first: they are the bulk of the traffic.
    float4 st[RPT];
#pragma unroll
    for (int r = 0; r < RPT; r++) st[r] = Sh[(size_t)(rg + r * RG) * (DV / 4) + cg];

    int flags = 0;
    float kq = 0.f;
    for (int i = tid; i < DK; i += NT) {
        float kv = to_f32(k[head * DK + i]);
        float qv = to_f32(q[head * DK + i]);
        float gv = g[head * DK + i];
        flags |= decay_flags(gv) | finite_flag(kv) | finite_flag(qv);
        s_k[i] = kv;
        s_q[i] = qv;
        s_a[i] = expf(gv);
        kq += kv * qv;
    }
    const float b = beta[head];
    if (tid == 0) flags |= finite_flag(b);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
    if ((tid & 31) == 0) s_kq[tid >> 5] = kq;
    __syncthreads();

    // S' = Diag(exp g) S, and partial sums of S'^T k and S'^T q.
    float pk[4] = {0.f, 0.f, 0.f, 0.f}, pq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int r = 0; r < RPT; r++) {
        const int i = rg + r * RG;
        const float a = s_a[i], ki = s_k[i], qi = s_q[i];
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
        s_red[0][rg][cg * 4 + c] = pk[c];
        s_red[1][rg][cg * 4 + c] = pq[c];
    }
    __syncthreads();

    // Column totals; every thread needs u for its own four columns.
    float kqt = 0.f;
#pragma unroll
    for (int w = 0; w < NW; w++) kqt += s_kq[w];
    float u[4];
#pragma unroll
    for (int c = 0; c < 4; c++) {
        const int j = cg * 4 + c;
        float kvj = 0.f, qvj = 0.f;
#pragma unroll
        for (int w = 0; w < RG; w++) {
            kvj += s_red[0][w][j];
            qvj += s_red[1][w][j];
        }
        const float vj = to_f32(v[head * DV + j0 + j]);
        flags |= finite_flag(vj);
        u[c] = b * (vj - kvj);
        if (rg == 0) o[head * DV + j0 + j] = from_f32<TIn>(qvj + u[c] * kqt);
    }

    // S = S' + k u^T, written back in place.
#pragma unroll
    for (int r = 0; r < RPT; r++) {
        const float ki = s_k[rg + r * RG];
        st[r].x += ki * u[0];
        st[r].y += ki * u[1];
        st[r].z += ki * u[2];
        st[r].w += ki * u[3];
        Sh[(size_t)(rg + r * RG) * (DV / 4) + cg] = st[r];
    }
    report_flags(d_status, flags);
}

template <typename TIn, int D>
cudaError_t launch_t(const DecodeArgs& a) {
    constexpr int DVS = D / 2, NT = D;  // two CTAs per head, 16 rows x 4 columns per thread
    const unsigned grid = (unsigned)((long long)a.N * a.H * (D / DVS));
    // a step of a decode loop: its launch overlaps the end of the previous one
    return launch_dependent(kda_decode_kernel<TIn, D, D, DVS, NT>, dim3(grid), dim3(NT), 0,
                            a.stream, static_cast<const TIn*>(a.q), static_cast<const TIn*>(a.k),
                            static_cast<const TIn*>(a.v), a.g, a.beta, a.S,
                            static_cast<TIn*>(a.o), a.d_status);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, kda_dtype_t io) {
    if (io == KDA_BF16) return a.dk == 128 ? launch_t<__nv_bfloat16, 128>(a)
                                           : launch_t<__nv_bfloat16, 64>(a);
    return a.dk == 128 ? launch_t<float, 128>(a) : launch_t<float, 64>(a);
}

}  // namespace kda
