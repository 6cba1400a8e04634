// KDA chunked forward on CUDA cores (fp32 arithmetic throughout).
//
// This is the high-accuracy path (fp32 inputs and outputs). It evaluates the
// same chunked algebra as the tensor-core path, with 16-token decay tiles,
// only on FFMA instead of MMA.
//
// Chunked form. The orkas.ai page "Kimi K3 architecture" (section "A lower
// bound that deleted a GPU code path") says the blockwise evaluation divides
// by the accumulated decay and that, with g >= -5, a 16-token tile's
// cumulative log-decay stays in (-80, 0], so its reciprocal (< e^80) is
// representable and the diagonal tiles need no pairwise special path. The
// pages give no formulas; the algebra below is derived from the recurrence
//     S_t = (I - b_t k_t k_t^T) Diag(e^{g_t}) S_{t-1} + b_t k_t v_t^T,  o_t = S_t^T q_t.
// For a chunk of C tokens with incoming state S0 and G_r = sum_{s<=r} g_s
// (per channel, relative to the chunk start):
//     (I + A) U = Diag(b) (V - Kt S0),   A_rs = b_r sum_c k_rc k_sc e^{G_rc - G_sc}  (s < r)
//     T = (I + A)^-1,  W = T Diag(b) Kt,  Ut = T Diag(b) V,  U = Ut - W S0
//     O = Qt S0 + P U,  P_rs = sum_c q_rc k_sc e^{G_rc - G_sc}  (s <= r)
//     S_C = Diag(e^{G_C}) S0 + Kb^T U
// with Kt_r = k_r e^{G_r}, Qt_r = q_r e^{G_r}, Kb_s = k_s e^{G_C - G_s}.
// The decay ratio e^{G_rc - G_sc} is split at the start of r's 16-token tile
// a (anchor a-): e^{G_r - G_a-} <= 1 on the row side and, on the column side,
//   s in the same tile:     e^{G_a- - G_s}  in [1, e^80)   (the bounded reciprocal)
//   s in an earlier tile b: e^{G_a- - G_b+} e^{G_b+ - G_s}, both <= 1,
// where b+ is the end of tile b. Each factor is computed from differences of
// G, never as a quotient of two decays, so nothing overflows or loses
// precision to denormals.
//
// One CTA owns one (b, h, dv-slice); the state slice S[dk][DVS] stays in
// shared memory for the whole sequence. Rows past T are zero-padded with
// g = 0, beta = 0, which makes them exact no-ops.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kTile = 16;

template <int DK, int DVS, int C>
struct SimtSmem {
    static constexpr int LDK = DK + 1;  // padded rows: conflict-free column walks
    static constexpr int LDV = DVS + 1;
    static constexpr int LDC = C + 1;
    static constexpr int NTL = C / kTile;
    float K[C * LDK];   // k, then Kp = k e^{G-Ga}, then Kt
    float Q[C * LDK];   // q, then Qp, then Qt
    float G[C * LDK];   // cumulative log-decay G
    float Km[C * LDK];  // k e^{Ga-G} (same-tile column operand), then W
    float Ke[C * LDK];  // k e^{Ge-G} (earlier-tile column operand), then Kb
    float V[C * LDV];   // v slice, then U
    float Ut[C * LDV];  // T Diag(b) V
    float A[C * LDC];   // strict lower A (row-scaled by beta)
    float P[C * LDC];   // lower P incl. diagonal
    float Tm[C * LDC];  // T Diag(beta)
    float S[DK * LDV];  // state slice
    float Ga[NTL][DK];  // G just before each tile (anchor)
    float Ge[NTL][DK];  // G at the last row of each tile
    float R[NTL][NTL][DK];  // e^{Ga[a] - Ge[b]}, b < a
    float Ea[NTL][DK];  // e^{Ga[a]}
    float Ec[NTL][DK];  // e^{G_C - Ge[b]}
    float lam[DK];      // e^{G_C}
    float beta[C];
};

template <typename TIn, int DK, int DVS, int C, int NT>
__global__ void __launch_bounds__(NT, 1)
    kda_chunk_simt_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k,
                          const TIn* __restrict__ v, const float* __restrict__ g,
                          const float* __restrict__ beta, const float* __restrict__ h0,
                          TIn* __restrict__ o, float* __restrict__ hT, int T, int H, int DV,
                          int* __restrict__ d_status, float* __restrict__ ckpt, int ckpt_every) {
    using Sm = SimtSmem<DK, DVS, C>;
    constexpr int LDK = Sm::LDK, LDV = Sm::LDV, LDC = Sm::LDC, NTL = Sm::NTL;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Sm& sm = *reinterpret_cast<Sm*>(smem_raw);

    const int tid = threadIdx.x;
    const int j0 = blockIdx.x * DVS;  // dv slice start
    const int h = blockIdx.y, b = blockIdx.z;
    const size_t st_base = ((size_t)b * H + h) * DK * DV;

    // Incoming state.
    for (int idx = tid; idx < DK * DVS; idx += NT) {
        const int i = idx / DVS, j = idx % DVS;
        sm.S[i * LDV + j] = h0 ? h0[st_base + (size_t)i * DV + j0 + j] : 0.f;
    }

    int flags = 0;
    for (int t0 = 0; t0 < T; t0 += C) {
        const int L = min(C, T - t0);
        __syncthreads();  // previous chunk done with every buffer
        // ---- stage the chunk (zero-padded past T) ----
        for (int idx = tid; idx < C * DK; idx += NT) {
            const int r = idx / DK, c = idx % DK;
            float kv = 0.f, qv = 0.f, gv = 0.f;
            if (r < L) {
                const size_t gi = (((size_t)b * T + t0 + r) * H + h) * DK + c;
                kv = to_f32(k[gi]);
                qv = to_f32(q[gi]);
                gv = g[gi];
                flags |= decay_flags(gv);
            }
            sm.K[r * LDK + c] = kv;
            sm.Q[r * LDK + c] = qv;
            sm.G[r * LDK + c] = gv;
        }
        for (int idx = tid; idx < C * DVS; idx += NT) {
            const int r = idx / DVS, j = idx % DVS;
            sm.V[r * LDV + j] =
                r < L ? to_f32(v[(((size_t)b * T + t0 + r) * H + h) * DV + j0 + j]) : 0.f;
        }
        for (int r = tid; r < C; r += NT) {
            float bv = r < L ? beta[((size_t)b * T + t0 + r) * H + h] : 0.f;
            flags |= finite_flag(bv);
            sm.beta[r] = bv;
        }
        __syncthreads();

        // ---- cumulative log-decay per channel, tile anchors ----
        for (int c = tid; c < DK; c += NT) {
            float acc = 0.f;
            for (int a = 0; a < NTL; a++) {
                sm.Ga[a][c] = acc;
                for (int r = a * kTile; r < (a + 1) * kTile; r++) {
                    acc += sm.G[r * LDK + c];
                    sm.G[r * LDK + c] = acc;
                }
                sm.Ge[a][c] = acc;
            }
            sm.lam[c] = expf(acc);
            for (int a = 0; a < NTL; a++) {
                sm.Ea[a][c] = expf(sm.Ga[a][c]);
                sm.Ec[a][c] = expf(acc - sm.Ge[a][c]);
                for (int bb = 0; bb < a; bb++) sm.R[a][bb][c] = expf(sm.Ga[a][c] - sm.Ge[bb][c]);
            }
        }
        __syncthreads();

        // ---- decay-scaled operands ----
        for (int idx = tid; idx < C * DK; idx += NT) {
            const int r = idx / DK, c = idx % DK, a = r / kTile;
            const float G = sm.G[r * LDK + c];
            const float ga = sm.Ga[a][c], ge = sm.Ge[a][c];
            const float kv = sm.K[r * LDK + c];
            const float ep = expf(G - ga);            // <= 1
            sm.Km[r * LDK + c] = kv * expf(ga - G);   // in [1, e^80) times k
            sm.Ke[r * LDK + c] = kv * expf(ge - G);   // <= 1 times k
            sm.K[r * LDK + c] = kv * ep;
            sm.Q[r * LDK + c] *= ep;
        }
        __syncthreads();

        // ---- Gram matrices A (strict lower, row-scaled by beta) and P (lower) ----
        for (int p = tid; p < C * C; p += NT) {
            const int r = p / C, s = p % C;
            float accA = 0.f, accP = 0.f;
            if (s <= r) {
                const int a = r / kTile, bt = s / kTile;
                const float* kr = &sm.K[r * LDK];
                const float* qr = &sm.Q[r * LDK];
                if (a == bt) {
                    const float* ks = &sm.Km[s * LDK];
#pragma unroll 8
                    for (int c = 0; c < DK; c++) {
                        accA += kr[c] * ks[c];
                        accP += qr[c] * ks[c];
                    }
                } else {
                    const float* ks = &sm.Ke[s * LDK];
                    const float* rr = sm.R[a][bt];
#pragma unroll 8
                    for (int c = 0; c < DK; c++) {
                        const float x = ks[c] * rr[c];
                        accA += kr[c] * x;
                        accP += qr[c] * x;
                    }
                }
                accA = s < r ? accA * sm.beta[r] : 0.f;
            }
            sm.A[r * LDC + s] = accA;
            sm.P[r * LDC + s] = accP;
        }
        __syncthreads();

        // ---- T = (I + A)^-1 by forward substitution, one column per thread;
        //      stored as T Diag(beta) ----
        for (int s = tid; s < C; s += NT) {
            float col[C];
#pragma unroll
            for (int r = 0; r < C; r++) col[r] = 0.f;
            col[s] = 1.f;
            for (int r = s + 1; r < C; r++) {
                float acc = 0.f;
                for (int m = s; m < r; m++) acc += sm.A[r * LDC + m] * col[m];
                col[r] = -acc;
            }
            const float bs = sm.beta[s];
#pragma unroll
            for (int r = 0; r < C; r++) sm.Tm[r * LDC + s] = col[r] * bs;
        }
        // Kt = Kp e^{Ga}, Qt = Qp e^{Ga}, Kb = Ke e^{G_C - Ge} (products of factors <= 1).
        for (int idx = tid; idx < C * DK; idx += NT) {
            const int r = idx / DK, c = idx % DK, a = r / kTile;
            sm.K[r * LDK + c] *= sm.Ea[a][c];
            sm.Q[r * LDK + c] *= sm.Ea[a][c];
            sm.Ke[r * LDK + c] *= sm.Ec[a][c];
        }
        __syncthreads();

        // ---- W = T Diag(b) Kt (into Km), Ut = T Diag(b) V ----
        for (int idx = tid; idx < C * DK; idx += NT) {
            const int r = idx / DK, c = idx % DK;
            float acc = 0.f;
            for (int s = 0; s <= r; s++) acc += sm.Tm[r * LDC + s] * sm.K[s * LDK + c];
            sm.Km[r * LDK + c] = acc;
        }
        for (int idx = tid; idx < C * DVS; idx += NT) {
            const int r = idx / DVS, j = idx % DVS;
            float acc = 0.f;
            for (int s = 0; s <= r; s++) acc += sm.Tm[r * LDC + s] * sm.V[s * LDV + j];
            sm.Ut[r * LDV + j] = acc;
        }
        __syncthreads();

        // ---- U = Ut - W S0 (into V) ----
        for (int idx = tid; idx < C * DVS; idx += NT) {
            const int r = idx / DVS, j = idx % DVS;
            float acc = sm.Ut[r * LDV + j];
            for (int i = 0; i < DK; i++) acc -= sm.Km[r * LDK + i] * sm.S[i * LDV + j];
            sm.V[r * LDV + j] = acc;
        }
        __syncthreads();

        // ---- O = Qt S0 + P U ----
        for (int idx = tid; idx < C * DVS; idx += NT) {
            const int r = idx / DVS, j = idx % DVS;
            if (r >= L) continue;
            float acc = 0.f;
            for (int i = 0; i < DK; i++) acc += sm.Q[r * LDK + i] * sm.S[i * LDV + j];
            for (int s = 0; s <= r; s++) acc += sm.P[r * LDC + s] * sm.V[s * LDV + j];
            flags |= finite_flag(acc);  // a NaN or Inf in q, k or v reaches some output
            o[(((size_t)b * T + t0 + r) * H + h) * DV + j0 + j] = from_f32<TIn>(acc);
        }
        __syncthreads();

        // ---- S = Diag(e^{G_C}) S0 + Kb^T U ----
        for (int idx = tid; idx < DK * DVS; idx += NT) {
            const int i = idx / DVS, j = idx % DVS;
            float acc = sm.lam[i] * sm.S[i * LDV + j];
            for (int s = 0; s < C; s++) acc += sm.Ke[s * LDK + i] * sm.V[s * LDV + j];
            sm.S[i * LDV + j] = acc;
        }
        if (ckpt && (t0 + C) % ckpt_every == 0 && t0 + C <= T) {  // sparse state checkpoint
            __syncthreads();
            const int n_ckpt = T / ckpt_every, jc = (t0 + C) / ckpt_every - 1;
            float* dst = ckpt + (((size_t)b * H + h) * n_ckpt + jc) * DK * DV;
            for (int idx = tid; idx < DK * DVS; idx += NT) {
                const int i = idx / DVS, j = idx % DVS;
                dst[(size_t)i * DV + j0 + j] = sm.S[i * LDV + j];
            }
        }
    }
    __syncthreads();
    report_flags(d_status, flags);
    if (hT) {
        for (int idx = tid; idx < DK * DVS; idx += NT) {
            const int i = idx / DVS, j = idx % DVS;
            hT[st_base + (size_t)i * DV + j0 + j] = sm.S[i * LDV + j];
        }
    }
}

template <typename TIn, int DK>
cudaError_t launch_t(const ChunkFwdArgs& a) {
    constexpr int C = 32, DVS = 64, NT = 256;
    using Sm = SimtSmem<DK, DVS, C>;
    auto kern = kda_chunk_simt_kernel<TIn, DK, DVS, C, NT>;
    const size_t smem = sizeof(Sm);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.dv / DVS, a.H, a.B);
    kern<<<grid, NT, smem, a.stream>>>(
        static_cast<const TIn*>(a.q), static_cast<const TIn*>(a.k), static_cast<const TIn*>(a.v),
        a.g, a.beta, a.h0, static_cast<TIn*>(a.o), a.hT, a.T, a.H, a.dv, a.d_status, a.ckpt,
        a.ckpt_every);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunk_fwd_simt(const ChunkFwdArgs& a, kda_dtype_t io) {
    if (io == KDA_BF16)
        return a.dk == 128 ? launch_t<__nv_bfloat16, 128>(a) : launch_t<__nv_bfloat16, 64>(a);
    return a.dk == 128 ? launch_t<float, 128>(a) : launch_t<float, 64>(a);
}

}  // namespace kda
