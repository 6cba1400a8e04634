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
//     o  = S^T q = S'^T q + u (k . q),
// evaluated with S'^T k = S^T (e^g k) and S'^T q = S^T (e^g q), so both
// reductions read the state before its decay.
//
// Layout. One warp per (sequence, head, 32-column slice of the value
// channels); the D / 32 warps of a head form one CTA and share its staged
// token vectors. Lane l owns columns j0 + 4 (l % 8) .. + 3 of rows
// (l / 8) * D/4 .. + D/4 - 1 in registers (32 float4 at D = 128) for all the
// sequence's tokens: the state is read once and written at most once. The
// reductions over the key channel finish inside the warp (two xor-shuffle
// steps across the four row groups), so the token loop has no barrier; the
// token vectors (e^g k, e^g q, k, e^g, v, beta, k . q) are staged in shared
// memory eight tokens at a time, with one barrier per eight tokens.
//
// A verify of at most eight drafts runs kda_verify_block_kernel instead: the
// block form of the recurrence reads only the incoming state, so the state
// streams through registers (see there).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kStage = 8;  // tokens staged per pass

// WANT_O: outputs are computed (verify, or commit with o); without them the
// reduction S^T (e^g q) is skipped. A verify leaves the state as it was, so
// its last token's update is skipped too.
template <typename TIn, int D, bool WANT_O>
__global__ void __launch_bounds__(D, 384 / D)
    kda_decode_multi_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k,
                            const TIn* __restrict__ v, const float* __restrict__ g,
                            const float* __restrict__ beta, float* __restrict__ S,
                            TIn* __restrict__ o, const int* __restrict__ ntok, int K, int H,
                            int commit, int* __restrict__ d_status) {
    constexpr int R = D / 4;    // state rows per thread
    constexpr int NW = D / 32;  // warps = 32-column value slices per head
    // Key-channel vectors keep four padding words after each row group's R
    // entries, so the four row groups' float4 reads fall on distinct banks.
    constexpr int LDP = D + 16;
    __shared__ __align__(16) float s_lk[kStage][LDP], s_lq[kStage][LDP], s_k[kStage][LDP],
        s_lam[kStage][LDP];
    __shared__ __align__(16) float s_v[kStage][D];
    __shared__ float s_kqp[kStage][NW], s_beta[kStage];

    pdl_wait();  // the kernel before it in the stream is done
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t head = blockIdx.x;  // n * H + h
    const int n = (int)(head / H), hh = (int)(head % H);
    const int cg = lane & 7, rg = lane >> 3;
    const int j = 32 * warp + 4 * cg;  // first of this thread's four value columns
    const int i0 = rg * R;             // first of its state rows
    const int p0 = rg * (R + 4);       // where they start in the padded vectors
    const int ptid = tid + (tid / R) * 4;
    int nt = K;
    if (ntok) nt = min(max(ntok[n], 0), K);
    if (nt == 0) return;
    float4* Sh = reinterpret_cast<float4*>(S + head * D * D + j);

    float4 st[R];
#pragma unroll
    for (int r = 0; r < R; r++) st[r] = Sh[(size_t)(i0 + r) * (D / 4)];

    int flags = 0;
    for (int t0 = 0; t0 < nt; t0 += kStage) {
        const int nb = min(kStage, nt - t0);
        if (t0 > 0) __syncthreads();  // the previous block's vectors are consumed
        // Stage: thread tid owns key channel (and value column) tid of each token.
        for (int tt = 0; tt < nb; tt++) {
            const size_t row = ((size_t)n * K + t0 + tt) * H + hh;
            const float kv = to_f32(k[row * D + tid]);
            const float qv = to_f32(q[row * D + tid]);
            const float gv = g[row * D + tid];
            const float vv = to_f32(v[row * D + tid]);
            flags |= decay_flags(gv) | finite_flag(kv) | finite_flag(qv) | finite_flag(vv);
            const float lam = expf(gv);
            s_k[tt][ptid] = kv;
            s_lam[tt][ptid] = lam;
            s_lk[tt][ptid] = lam * kv;
            s_lq[tt][ptid] = lam * qv;
            s_v[tt][tid] = vv;
            float kq = kv * qv;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
            if (lane == 0) s_kqp[tt][warp] = kq;
        }
        if (tid < nb) {
            const float b = beta[((size_t)n * K + t0 + tid) * H + hh];
            flags |= finite_flag(b);
            s_beta[tid] = b;
        }
        __syncthreads();

        for (int tt = 0; tt < nb; tt++) {
            // a = S^T (e^g k), b = S^T (e^g q) over this thread's rows
            float a[4] = {0.f, 0.f, 0.f, 0.f}, bq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int r4 = 0; r4 < R; r4 += 4) {
                const float4 lk = *reinterpret_cast<const float4*>(&s_lk[tt][p0 + r4]);
                const float4 lq = *reinterpret_cast<const float4*>(&s_lq[tt][p0 + r4]);
                const float lkv[4] = {lk.x, lk.y, lk.z, lk.w};
                const float lqv[4] = {lq.x, lq.y, lq.z, lq.w};
#pragma unroll
                for (int rr = 0; rr < 4; rr++) {
                    const float4 s4 = st[r4 + rr];
                    a[0] = fmaf(s4.x, lkv[rr], a[0]);
                    a[1] = fmaf(s4.y, lkv[rr], a[1]);
                    a[2] = fmaf(s4.z, lkv[rr], a[2]);
                    a[3] = fmaf(s4.w, lkv[rr], a[3]);
                    if (WANT_O) {
                        bq[0] = fmaf(s4.x, lqv[rr], bq[0]);
                        bq[1] = fmaf(s4.y, lqv[rr], bq[1]);
                        bq[2] = fmaf(s4.z, lqv[rr], bq[2]);
                        bq[3] = fmaf(s4.w, lqv[rr], bq[3]);
                    }
                }
            }
            // totals over the four row groups (lanes l, l ^ 8, l ^ 16, l ^ 24)
#pragma unroll
            for (int off = 8; off < 32; off <<= 1) {
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    a[c] += __shfl_xor_sync(0xffffffffu, a[c], off);
                    if (WANT_O) bq[c] += __shfl_xor_sync(0xffffffffu, bq[c], off);
                }
            }
            float kq = 0.f;
#pragma unroll
            for (int w = 0; w < NW; w++) kq += s_kqp[tt][w];
            const float bt = s_beta[tt];
            const float4 v4 = *reinterpret_cast<const float4*>(&s_v[tt][j]);
            const float vv[4] = {v4.x, v4.y, v4.z, v4.w};
            float u[4], ov[4];
#pragma unroll
            for (int c = 0; c < 4; c++) {
                u[c] = bt * (vv[c] - a[c]);
                ov[c] = bq[c] + u[c] * kq;
            }
            if (WANT_O && rg == (tt & 3)) {  // the four row groups take turns storing
                TIn* dst = o + (((size_t)n * K + t0 + tt) * H + hh) * D + j;
                if constexpr (sizeof(TIn) == 2) {
                    __nv_bfloat162 h0 = __floats2bfloat162_rn(ov[0], ov[1]);
                    __nv_bfloat162 h1 = __floats2bfloat162_rn(ov[2], ov[3]);
                    uint2 pk;
                    pk.x = *reinterpret_cast<uint32_t*>(&h0);
                    pk.y = *reinterpret_cast<uint32_t*>(&h1);
                    *reinterpret_cast<uint2*>(dst) = pk;
                } else {
                    *reinterpret_cast<float4*>(dst) = make_float4(ov[0], ov[1], ov[2], ov[3]);
                }
            }
            if (!commit && t0 + tt + 1 == nt) break;  // a verify needs no state after its last token
            // S = Diag(e^g) S + k u^T
#pragma unroll
            for (int r4 = 0; r4 < R; r4 += 4) {
                const float4 kk = *reinterpret_cast<const float4*>(&s_k[tt][p0 + r4]);
                const float4 ll = *reinterpret_cast<const float4*>(&s_lam[tt][p0 + r4]);
                const float kv[4] = {kk.x, kk.y, kk.z, kk.w};
                const float lv[4] = {ll.x, ll.y, ll.z, ll.w};
#pragma unroll
                for (int rr = 0; rr < 4; rr++) {
                    float4& s4 = st[r4 + rr];
                    s4.x = fmaf(lv[rr], s4.x, kv[rr] * u[0]);
                    s4.y = fmaf(lv[rr], s4.y, kv[rr] * u[1]);
                    s4.z = fmaf(lv[rr], s4.z, kv[rr] * u[2]);
                    s4.w = fmaf(lv[rr], s4.w, kv[rr] * u[3]);
                }
            }
        }
    }
    if (commit) {
#pragma unroll
        for (int r = 0; r < R; r++) Sh[(size_t)(i0 + r) * (D / 4)] = st[r];
    }
    report_flags(d_status, flags);
}

// Verify of up to KMAX draft tokens in the block form of the recurrence.
//
// A verify leaves the state as it was, and in the block form every reduction
// reads the incoming state S0 only:
//   Y_t = S0^T (k_t e^{G_t}),  Z_t = S0^T (q_t e^{G_t}),
//   A_ts = b_t sum_i k_t,i k_s,i e^{G_t,i - G_s,i} (s < t),
//   P_ts = sum_i q_t,i k_s,i e^{G_t,i - G_s,i} (s <= t),  T' = (I + A)^-1 Diag(b),
//   U = T' (V - Y),  O = Z + P U,
// (G_t = cumulative log-decay through draft token t; at most 8 x 5 = 40 in
// magnitude under the bound g >= -5, so e^{-G} stays far inside fp32). So the
// state streams through registers a few rows at a time instead of being held:
// fewer registers, more CTAs per SM, two multiply-adds per state element and
// token instead of four. Layout as in the per-token kernel: one warp per
// 32-column value slice, lane (rg, cg) rows rg D/4 .. + D/4 - 1, columns
// 4 cg .. + 3 of the slice.
template <typename TIn, int D, int KMAX>
__global__ void __launch_bounds__(D, KMAX <= 4 ? 6 : 3)
    kda_verify_block_kernel(const TIn* __restrict__ q, const TIn* __restrict__ k,
                            const TIn* __restrict__ v, const float* __restrict__ g,
                            const float* __restrict__ beta, const float* __restrict__ S,
                            TIn* __restrict__ o, const int* __restrict__ ntok, int K, int H,
                            int* __restrict__ d_status) {
    constexpr int R = D / 4;    // state rows per thread
    constexpr int NW = D / 32;  // warps
    constexpr int LDP = D + 16;
    constexpr int NPAIR = KMAX * (KMAX + 1) / 2;
    __shared__ __align__(16) float s_kt[KMAX][LDP];  // k e^{G}
    __shared__ __align__(16) float s_qt[KMAX][LDP];  // q e^{G}
    __shared__ __align__(16) float s_kh[KMAX][D];    // k e^{-G}
    __shared__ __align__(16) float s_v[KMAX][D];
    __shared__ float s_a[KMAX][KMAX], s_p[KMAX][KMAX], s_tp[KMAX][KMAX], s_beta[KMAX];

    pdl_wait();  // the kernel before it in the stream is done
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t head = blockIdx.x;  // n * H + h
    const int n = (int)(head / H), hh = (int)(head % H);
    const int cg = lane & 7, rg = lane >> 3;
    const int j = 32 * warp + 4 * cg;
    const int i0 = rg * R, p0 = rg * (R + 4);
    const int ptid = tid + (tid / R) * 4;
    int nt = K;
    if (ntok) nt = min(max(ntok[n], 0), K);
    if (nt == 0) return;
    int flags = 0;
    // The first rows of the state are requested before anything else.
    constexpr int GRP = 8;  // state rows per group of loads
    const float4* Sh = reinterpret_cast<const float4*>(S + head * D * D + j);
    float4 st[GRP];
#pragma unroll
    for (int rr = 0; rr < GRP; rr++) st[rr] = __ldcs(Sh + (size_t)(i0 + rr) * (D / 4));
    // ---- stage the draft tokens (thread = key channel / value column)
    {
        float G = 0.f;
#pragma unroll
        for (int t = 0; t < KMAX; t++) {
            if (t < nt) {
                const size_t row = ((size_t)n * K + t) * H + hh;
                const float kv = to_f32(k[row * D + tid]);
                const float qv = to_f32(q[row * D + tid]);
                const float gv = g[row * D + tid];
                const float vv = to_f32(v[row * D + tid]);
                flags |= decay_flags(gv) | finite_flag(kv) | finite_flag(qv) | finite_flag(vv);
                G += gv;
                const float e = expf(G);
                s_kt[t][ptid] = kv * e;
                s_qt[t][ptid] = qv * e;
                s_kh[t][tid] = kv * expf(-G);
                s_v[t][tid] = vv;
            }
        }
        if (tid < nt) {
            const float b = beta[((size_t)n * K + tid) * H + hh];
            flags |= finite_flag(b);
            s_beta[tid] = b;
        }
    }
    __syncthreads();
    // ---- Gram blocks: pair (t, s), s <= t, on warp (pair % NW), lanes split the channels
#pragma unroll
    for (int pi = warp; pi < NPAIR; pi += NW) {
        int t = 0;
        while ((t + 1) * (t + 2) / 2 <= pi) t++;
        const int s = pi - t * (t + 1) / 2;
        if (t < nt) {
            float a = 0.f, pq = 0.f;
#pragma unroll
            for (int c = lane; c < D; c += 32) {
                const float kh = s_kh[s][c];
                const int pc = c + (c / R) * 4;
                a = fmaf(s_kt[t][pc], kh, a);
                pq = fmaf(s_qt[t][pc], kh, pq);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                a += __shfl_xor_sync(0xffffffffu, a, off);
                pq += __shfl_xor_sync(0xffffffffu, pq, off);
            }
            if (lane == 0) {
                s_a[t][s] = a;
                s_p[t][s] = pq;
            }
        }
    }
    __syncthreads();  // Gram blocks from all warps
    // ---- T' = (I + A)^-1 Diag(b), column s by thread s (forward substitution)
    if (tid < nt) {
        const int s = tid;
        float col[KMAX];
#pragma unroll
        for (int t = 0; t < KMAX; t++) {
            float x = 0.f;
            if (t == s) {
                x = 1.f;
            } else if (t > s && t < nt) {
                const float bt = s_beta[t];
#pragma unroll
                for (int m = 0; m < KMAX; m++)
                    if (m >= s && m < t) x -= bt * s_a[t][m] * col[m];
            }
            col[t] = x;
        }
        const float bs = s_beta[s];
#pragma unroll
        for (int t = 0; t < KMAX; t++) s_tp[t][s] = t >= s ? col[t] * bs : 0.f;
    }
    // ---- the state streamed through registers: Y_t, Z_t over this thread's rows
    float y[KMAX][4], z[KMAX][4];
#pragma unroll
    for (int t = 0; t < KMAX; t++)
#pragma unroll
        for (int c = 0; c < 4; c++) y[t][c] = z[t][c] = 0.f;
#pragma unroll
    for (int r0 = 0; r0 < R; r0 += GRP) {
        if (r0 > 0) {
#pragma unroll
            for (int rr = 0; rr < GRP; rr++) st[rr] = __ldcs(Sh + (size_t)(i0 + r0 + rr) * (D / 4));
        }
#pragma unroll
        for (int t = 0; t < KMAX; t++) {
            if (t < nt) {
#pragma unroll
                for (int r4 = 0; r4 < GRP; r4 += 4) {
                    const float4 lk = *reinterpret_cast<const float4*>(&s_kt[t][p0 + r0 + r4]);
                    const float4 lq = *reinterpret_cast<const float4*>(&s_qt[t][p0 + r0 + r4]);
                    const float kk[4] = {lk.x, lk.y, lk.z, lk.w};
                    const float qq[4] = {lq.x, lq.y, lq.z, lq.w};
#pragma unroll
                    for (int rr = 0; rr < 4; rr++) {
                        const float4 s4 = st[r4 + rr];
                        y[t][0] = fmaf(s4.x, kk[rr], y[t][0]);
                        y[t][1] = fmaf(s4.y, kk[rr], y[t][1]);
                        y[t][2] = fmaf(s4.z, kk[rr], y[t][2]);
                        y[t][3] = fmaf(s4.w, kk[rr], y[t][3]);
                        z[t][0] = fmaf(s4.x, qq[rr], z[t][0]);
                        z[t][1] = fmaf(s4.y, qq[rr], z[t][1]);
                        z[t][2] = fmaf(s4.z, qq[rr], z[t][2]);
                        z[t][3] = fmaf(s4.w, qq[rr], z[t][3]);
                    }
                }
            }
        }
    }
    // totals over the four row groups (lanes l, l ^ 8, l ^ 16, l ^ 24)
#pragma unroll
    for (int t = 0; t < KMAX; t++) {
        if (t < nt) {
#pragma unroll
            for (int off = 8; off < 32; off <<= 1)
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    y[t][c] += __shfl_xor_sync(0xffffffffu, y[t][c], off);
                    z[t][c] += __shfl_xor_sync(0xffffffffu, z[t][c], off);
                }
        }
    }
    __syncthreads();  // T' from threads 0 .. nt - 1
    // ---- U = T' (V - Y), O = Z + P U for this thread's four columns
    float u[KMAX][4];
#pragma unroll
    for (int t = 0; t < KMAX; t++) {
#pragma unroll
        for (int c = 0; c < 4; c++) u[t][c] = 0.f;
        if (t < nt) {
#pragma unroll
            for (int s = 0; s < KMAX; s++) {
                if (s <= t) {
                    const float w = s_tp[t][s];
                    const float4 v4 = *reinterpret_cast<const float4*>(&s_v[s][j]);
                    u[t][0] = fmaf(w, v4.x - y[s][0], u[t][0]);
                    u[t][1] = fmaf(w, v4.y - y[s][1], u[t][1]);
                    u[t][2] = fmaf(w, v4.z - y[s][2], u[t][2]);
                    u[t][3] = fmaf(w, v4.w - y[s][3], u[t][3]);
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < KMAX; t++) {
        if (t < nt && rg == (t & 3)) {
            float ov[4] = {z[t][0], z[t][1], z[t][2], z[t][3]};
#pragma unroll
            for (int s = 0; s < KMAX; s++) {
                if (s <= t) {
                    const float pp = s_p[t][s];
#pragma unroll
                    for (int c = 0; c < 4; c++) ov[c] = fmaf(pp, u[s][c], ov[c]);
                }
            }
            TIn* dst = o + (((size_t)n * K + t) * H + hh) * D + j;
            if constexpr (sizeof(TIn) == 2) {
                __nv_bfloat162 h0 = __floats2bfloat162_rn(ov[0], ov[1]);
                __nv_bfloat162 h1 = __floats2bfloat162_rn(ov[2], ov[3]);
                uint2 pk;
                pk.x = *reinterpret_cast<uint32_t*>(&h0);
                pk.y = *reinterpret_cast<uint32_t*>(&h1);
                *reinterpret_cast<uint2*>(dst) = pk;
            } else {
                *reinterpret_cast<float4*>(dst) = make_float4(ov[0], ov[1], ov[2], ov[3]);
            }
        }
    }
    report_flags(d_status, flags);
}

template <typename TIn, int D>
cudaError_t launch_t(const MultiDecodeArgs& a) {
    const unsigned grid = (unsigned)((long long)a.N * a.H);
    if (!a.commit && a.o && a.K <= 8) {  // a verify of up to eight drafts: block form, state streamed
        auto vk = a.K <= 4 ? kda_verify_block_kernel<TIn, D, 4> : kda_verify_block_kernel<TIn, D, 8>;
        return launch_dependent(vk, dim3(grid), dim3(D), 0, a.stream,
                                static_cast<const TIn*>(a.q), static_cast<const TIn*>(a.k),
                                static_cast<const TIn*>(a.v), a.g, a.beta,
                                static_cast<const float*>(a.S), static_cast<TIn*>(a.o), a.ntok,
                                a.K, a.H, a.d_status);
    }
    auto kern = a.o ? kda_decode_multi_kernel<TIn, D, true> : kda_decode_multi_kernel<TIn, D, false>;
    return launch_dependent(kern, dim3(grid), dim3(D), 0, a.stream, static_cast<const TIn*>(a.q),
                            static_cast<const TIn*>(a.k), static_cast<const TIn*>(a.v), a.g,
                            a.beta, a.S, static_cast<TIn*>(a.o), a.ntok, a.K, a.H, a.commit,
                            a.d_status);
}

}  // namespace

cudaError_t launch_decode_multi(const MultiDecodeArgs& a, kda_dtype_t io) {
    if (io == KDA_BF16) return a.dk == 128 ? launch_t<__nv_bfloat16, 128>(a)
                                           : launch_t<__nv_bfloat16, 64>(a);
    return a.dk == 128 ? launch_t<float, 128>(a) : launch_t<float, 64>(a);
}

}  // namespace kda
