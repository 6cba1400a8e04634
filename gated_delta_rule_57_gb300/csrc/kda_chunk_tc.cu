// KDA chunked forward on the Blackwell tensor cores (tcgen05 + TMEM + TMA),
// bf16 inputs/outputs, fp32 state, dk = dv = 128, chunks of C = 64 tokens
// split into four 16-token decay tiles.
//
// Method. The orkas.ai page "Kimi K3 architecture" (section "A lower bound
// that deleted a GPU code path") says the blockwise evaluation of the KDA
// state divides by the accumulated decay, that tiles of 16 tokens are used,
// and that with the log-decay bounded below by -5 the reciprocal decay over
// one tile stays below e^80, inside the bf16 range, so the diagonal tiles use
// the same dense matrix product as every other tile. This kernel does exactly
// that: inside a tile the column operand carries the reciprocal decay
// k_s e^{G_a- - G_s} (at most e^80 |k|) and goes through the same tcgen05
// MMA as the off-diagonal tiles; there is no pairwise path.
//
// Chunk algebra (derived from S_t = (I - b k k^T) Diag(e^g) S_{t-1} + b k v^T,
// o_t = S_t^T q_t; G = in-chunk cumulative log-decay, S0 = incoming state):
//   A_rs = b_r sum_c k_rc k_sc e^{G_rc-G_sc} (s<r),  P_rs = sum_c q_rc k_sc e^{G_rc-G_sc} (s<=r)
//   T' = (I + A)^-1 Diag(b),  Kt = k e^{G},  Qt = q e^{G},  Kb = k e^{G_C - G}
//   W = T' Kt,  Ut = T' V,  U = Ut - W S0,  O = Qt S0 + P U,  S_C = Diag(e^{G_C}) S0 + Kb^T U.
// Since W S0 = T' (Kt S0), the state enters only through Y = Kt S0 and
// Qt S0, which need neither the Gram matrices nor the solve. The state is kept
// transposed in tensor memory (lane = value channel j, column = key channel
// i), so its bf16 copy, V - Y and U serve as A operands straight from TMEM
// (two bf16 per 32-bit column). As 128-row MMAs (D^T = A B^T):
//   round 1  Gram blocks  [Kp; Qp] * [Km_0; Km_1; Km_2; Km_3]^T   (N = 16+32+48+64)
//   round 2  D1[:, 0:64] = V^T I (A = the v tile, MN-major; I a constant
//            identity), then D1 += S0^T [-Kt; Qt]^T -> [(V - Y)^T | (Qt S0)^T]
//            (A = S0^T in TMEM; under the solve)
//            (V - Y)^T -> bf16 A operand in TMEM (under the solve as well)
//   round 3  D1[:, 0:64] = (V - Y)^T T'^T -> U^T                  (A = (V - Y)^T in TMEM)
//   round 4  S^T += U^T Kb                 (S^T pre-scaled by e^{G_C} per key channel)
//            D1[:, 64:128] += U^T P^T      -> O^T = (Qt S0 + P U)^T   (A = U^T in TMEM)
// O^T is read out while the next chunk's round 1 runs, staged in shared
// memory as bf16 rows and written to o by one TMA store.
//
// Execution. One CTA per (b, h) sequence, 512 threads (four warps per TMEM
// lane quarter), ~226 KB of shared memory (one CTA per SM), 480 TMEM columns:
// the fp32 state stays in tensor memory for the whole sequence. When B * H
// sequences would leave a partly filled last wave, one CTA per SM instead
// runs an equal share of chunk steps over the sequences laid end to end (the
// balanced schedule, see TcParams); a sequence split between two CTAs passes
// its state through global memory once. Inputs arrive
// by TMA with the 128-byte swizzle (q, k, v in the layout the MMA descriptors
// expect; g in 32-channel blocks); the next chunk's g, q/k, v and beta are
// prefetched as soon as their buffers are free. Issuing a tcgen05.mma keeps
// the issuing thread busy for about the product's duration, so the rounds sit
// on warps whose own results are needed only later in the chunk: warp 15
// issues rounds 1 and 4 (and the next g tile), warp 12, which has no readout
// rows, round 2 and the O store, thread 0 round 3 (every warp waits for it).
// Completion is signalled through mbarriers whose waits are
// bounded (timeout -> KDA_DEV_TIMEOUT). A CTA barrier stands only where a
// phase reads other warps' results. The decay scan, the decay constants and
// the operand build need none: each warp owns eight channels of all four
// tiles (a lane scans one channel of one tile in registers), so tile totals
// and constants stay inside the warp, and it stores its Kt, Qt and Kb rows
// as it builds them. Round 1 waits on an arrive-only mbarrier.
// Intermediates never leave the SM: the kernel reads each input once and
// writes o (and hT) once. The <true> instantiation also runs the passes of
// the time-segmented evaluation and of a sequence split across devices (see
// TcParams).
#include <cudaTypedefs.h>

#include "kda_internal.cuh"
#include "sm100_ptx.cuh"

namespace kda {
namespace {

using namespace ptx;

constexpr int kC = 64;          // chunk length
constexpr int kD = 128;         // dk = dv
constexpr int kThreads = 512;   // 16 warps: 4 per TMEM lane quarter
// Rounds 1 and 4 and the next g tile are issued by warp 15 (issuing keeps a
// thread busy for about the MMA's duration; warp 15's other results are
// needed only late in the chunk).
constexpr int kIssueThread = kThreads - 32;
// Round 2 and the O store: warp 12, which has no readout rows and waits for
// round 2 itself.
constexpr int kR2Thread = 384;
// The next chunk's q/k and v tiles are requested by warp 10, idle in the solve.
constexpr int kTmaThread = 320;
constexpr float kLog2e = 1.4426950408889634f;

// Shared memory map (bytes from a 1024-aligned base).
constexpr uint32_t OFF_G = 0;          // g: 4 blocks of 32 channels, SW128; then tile totals and
                                       // decay constants (each warp in its own 8 channels' chunks)
constexpr uint32_t OFF_KQP = 32768;    // [k; q] -> [Kp; Qp], SW128, 128 rows x 128
constexpr uint32_t OFF_KM = 65536;     // Km windows (160 rows x 128) | solve scratch
constexpr uint32_t OFF_V = 106496;     // v, SW128, 64 rows x 128 (MN-major A of the V^T copy)
constexpr uint32_t OFF_A0 = 122880;    // [T'; P], SW128 128 x 64 (K-major B of rounds 3, 4)
constexpr uint32_t OFF_KB = 139264;    // Kb of even chunks, SW128 64 x 128 (MN-major B)
constexpr uint32_t OFF_AKQ = 155648;   // [Kt; Qt], SW128 128 x 128 (K-major B of round 2)
constexpr uint32_t OFF_KB1 = 188416;   // Kb of odd chunks
constexpr uint32_t OFF_OST = 204800;   // O rows of a chunk, bf16 [64][128] (TMA store source)
constexpr uint32_t OFF_BETA = 221184;  // fp32 [64]
static_assert(OFF_OST + 64 * 256 <= OFF_BETA, "O staging overlaps beta");
constexpr uint32_t OFF_LAM = 221440;   // fp32 [128]  e^{G_C}
constexpr uint32_t OFF_I = 222208;     // identity 64 x 64 bf16, SW128 K-major (B of the V^T copy)
static_assert(OFF_I % 1024 == 0 && OFF_I >= OFF_LAM + 512, "identity tile misplaced");
constexpr uint32_t SMEM_BYTES = OFF_I + 8192 + 1024;
// aliases inside OFF_KM (solve scratch lives between round 1 and the end of
// the solve)
constexpr int LDA = 68;  // fp32 A: TF32 fragment loads (bank 4g + t) and float4 row stores conflict-free
constexpr int LDT = 68;  // fp32 T: TF32 A-fragment loads conflict-free (B-fragment loads 2-way)
constexpr uint32_t OFF_FA = OFF_KM;                 // fp32 A [64][LDA]
constexpr uint32_t OFF_FT = OFF_FA + 64 * LDA * 4;  // fp32 T [64][LDT]
constexpr uint32_t OFF_MS = OFF_FT + 64 * LDT * 4;  // fp32 level-2 slabs, 4 warps x [16][8]
constexpr int KM_ROWS = 160;                  // windows of 16, 32, 48, 64 rows
__host__ __device__ __forceinline__ constexpr int win_row(int a) { return 8 * a * (a + 1); }
static_assert(OFF_MS + 4 * 128 * 4 <= OFF_V, "solve scratch overflows the window buffer");
static_assert(LDA % 4 == 0 && LDT % 4 == 0 && OFF_FA % 16 == 0 && OFF_FT % 16 == 0,
              "ldmatrix rows must start on 16-byte boundaries");

// TMEM columns: the transposed state, round 2/3/4 accumulators (D1), the
// Gram round's accumulator (SCR), and bf16 A operands (AUX: S0^T, then
// (V - Y)^T in columns 0..31 and U^T in 32..63).
constexpr uint32_t TM_S = 0, TM_D1 = 128, TM_SCR = 256, TM_AUX = 416, TM_COLS = 512;

enum { BAR_QK = 0, BAR_G = 1, BAR_V = 2, BAR_MMA = 3, BAR_R4 = 4, BAR_R2 = 5, BAR_P1 = 6, BAR_GP = 7, NBAR = 8 };

struct TcParams {
    const float* beta;
    const float* h0;
    __nv_bfloat16* o;
    float* hT;
    int T, H;
    int* d_status;
    float* ckpt;    // [B, H, n_ckpt, dk, dv] or null
    int ck_chunks;  // chunks between checkpoints
    int n_ckpt;
    // Segmented evaluation of long sequences (pass 0: one CTA per whole
    // sequence). Segment 0 spans lead * seg_chunks chunks, every later one
    // seg_chunks. Pass 1: CTA i < BH runs segment 0 of sequence i from h0
    // (the long runs start first), the next BH * (nseg - 1) CTAs segments
    // 1.. from a zero state, each writing o and its final state to ws_s0; the
    // last BH * (nseg - 1) CTAs run segments 1.. from the identity with v = 0,
    // leaving the segment transition in ws_m. Pass 2: segments 1.. again from
    // their incoming state ws_sin with v = 0, adding their outputs to o.
    // Whole-slice passes (one CTA per sequence, all its chunks), for a
    // sequence split across devices: pass 3 runs from the identity with
    // v = 0 and writes the slice's transition to ws_m[bh]; pass 4 runs from
    // ws_sin[bh] with v = 0 and adds its outputs to o.
    int pass, nseg, seg_chunks, lead, BH;
    // Device-planned split (passes 1 and 2): {nseg, seg_chunks, lead} are read
    // from here instead of the fields above, and the CTAs past the plan's
    // tasks leave at once (the grid is sized for the largest plan).
    const int* plan;
    // Balanced schedule of the whole-sequence kernel (bal_W > 0): CTA i covers
    // chunk steps [i bal_W, (i + 1) bal_W) of the sequences laid end to end
    // (bal_W >= the chunks of one sequence); a sequence split between two CTAs
    // hands its state over through bal_states[bh] and bal_flags[bh] (zeroed
    // before the launch; all CTAs are resident: cooperative launch).
    int bal_W;
    float* bal_states;  // [BH][dk][dv]
    int* bal_flags;     // [BH]
    float* ws_s0;         // [BH][nseg][dk][dv]
    float* ws_m;          // [BH][nseg - 1][dk][dk]
    const float* ws_sin;  // [BH][nseg - 1][dk][dv]
};

// 2^x on the SFU (ex2.approx, flush-to-zero). Arguments here are log2-decays
// in [-116, 116]; results below 2^-126 are decays too small to matter.
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint4 pack8(const float* x) {
    uint4 u;
    u.x = pack_bf16(x[0], x[1]);
    u.y = pack_bf16(x[2], x[3]);
    u.z = pack_bf16(x[4], x[5]);
    u.w = pack_bf16(x[6], x[7]);
    return u;
}
// bf16 is the upper half of an fp32 word: widening is a shift or a mask.
__device__ __forceinline__ void unpack8(uint4 u, float* x) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        x[2 * i] = __uint_as_float(w[i] << 16);
        x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Two 16-column TMEM loads (32x32b) under a single wait.
__device__ __forceinline__ void tmem_ld16x2(uint32_t ta, uint32_t tb, float* va, float* vb) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%33];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(ta), "r"(tb)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; i++) {
        va[i] = __uint_as_float(r[i]);
        vb[i] = __uint_as_float(r[16 + i]);
    }
}

// D[tmem] (+)= A[tmem] * B[smem]: A is M lanes x K, two bf16 per 32-bit column
// (k = 2c in the low half of column c), so a K = 16 step advances 8 columns.
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
        : "memory");
}
// 16 columns at ta and 32 at tb (32x32b) under a single wait.
__device__ __forceinline__ void tmem_ld16_32(uint32_t ta, uint32_t tb, float* va, float* vb) {
    uint32_t r[48];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%48];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
        "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47}, [%49];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
          "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
          "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47])
        : "r"(ta), "r"(tb)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; i++) va[i] = __uint_as_float(r[i]);
#pragma unroll
    for (int i = 0; i < 32; i++) vb[i] = __uint_as_float(r[16 + i]);
}
// Shared -> global tiled bulk copy (4-D map), tracked as a bulk group.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, const void* src, int c0, int c1,
                                             int c2, int c3) {
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];\n\t"
        "cp.async.bulk.commit_group;" ::"l"(reinterpret_cast<uint64_t>(map)),
        "r"(smem_addr(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
        : "memory");
}
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Handoff flag of the balanced schedule (GPU-scope acquire / release).
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu(int* p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Two bf16 (a in the low half) as the fp32 bit pattern tcgen05.st takes.
__device__ __forceinline__ float pack2f(float a, float b) { return __uint_as_float(pack_bf16(a, b)); }

// CTA barrier among `count` threads (whole warps) on named barrier `id` (1..15).
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// 8 consecutive bf16 (c0..c0+7, c0 % 8 == 0) of row r of an SW128 tile.
__device__ __forceinline__ void st_row8(unsigned char* tile, int r, int c0, int R,
                                        const float* x) {
    *reinterpret_cast<uint4*>(tile + sw128_offset(r, c0, R)) = pack8(x);
}

// Descriptors for the two operand orientations of an SW128 tile with R rows;
// k-step kk covers 16 elements of K. The start address is the low 14-bit
// field (in 16-byte units), so advancing an operand is a plain add.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t base) {
    return sdesc_sw128(base, 16, 1024);
}
__device__ __forceinline__ uint64_t kstep_kmajor(int R, int kk) {
    return (uint64_t)(((uint32_t)(kk >> 2) * (uint32_t)R * 128u + (uint32_t)(kk & 3) * 32u) >> 4);
}
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t base, int R) {
    return sdesc_sw128(base, (uint32_t)R * 128u, 1024);
}
__device__ __forceinline__ uint64_t kstep_mnmajor(int kk) { return (uint64_t)(kk * 128); }

// Warp-level TF32 MMA (m16n8k8, fp32 accumulate) for the 16-row blocks of
// the triangular inverse: tcgen05 needs M >= 64, these products are 16 x 16.
// Fragment ownership (g = lane / 4, t = lane % 4): A rows g, g+8 and columns
// t, t+4; B rows t, t+4 and column g; D rows g, g+8 and columns 2t, 2t+1.
// Operands are passed as their fp32 bits: the tensor core reads the TF32
// fields and drops the low 13 mantissa bits (round toward zero, relative
// error < 2^-10, below the bf16 rounding T' gets afterwards), which saves a
// conversion per element on these instruction-bound steps.
__device__ __forceinline__ uint32_t to_tf32(float x) { return __float_as_uint(x); }
// The A fragment of one m16n8k8 TF32 MMA (rows R0.., columns K0.. of a
// row-major fp32 matrix with leading dimension ld) in one ldmatrix.x4: seen as
// b16 pairs, matrix j of the four 8x4-word tiles hands thread i the word at
// (i / 4, i % 4), i.e. a[0..3] = (g, t), (g + 8, t), (g, t + 4), (g + 8, t + 4).
// Rows must start on 16-byte boundaries (ld and K0 multiples of 4).
__device__ __forceinline__ void ldsm_a_tf32(const float* m, int ld, int R0, int K0, int lane,
                                            uint32_t* a) {
    const int mat = lane >> 3, rr = lane & 7;
    const float* p = m + (R0 + rr + 8 * (mat & 1)) * ld + K0 + 4 * (mat >> 1);
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
                 : "r"(smem_addr(p))
                 : "memory");
}
__device__ __forceinline__ void mma_tf32(float* d, const uint32_t* a, const uint32_t* b) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Blocked triangular inverse T = (I + A)^-1 over 16-row blocks, merged as a
// tree: with the diagonal blocks T_ii known,
//   level 2:  T_10 = -T_11 A_10 T_00          T_32 = -T_33 A_32 T_22
//   level 3:  T_[23][01] = -T_[23][23] A_[23][01] T_[01][01]   (32 x 32 blocks)
// Each level is two dependent 16-row products on the TF32 tensor path; a warp
// computes the slab of the inner product that its own output tile needs into
// private shared memory, so only the levels are separated by CTA barriers.
// Blocks of T above the diagonal are never read; every finished block also
// goes out as T' = T Diag(beta) in bf16.
__device__ __forceinline__ void store_tprime(unsigned char* TP, const float* sbeta, int r, int n,
                                             const float* acc) {
    const float b0 = sbeta[n], b1 = sbeta[n + 1];
    *reinterpret_cast<uint32_t*>(TP + sw128_offset(r, n, 128)) =
        pack_bf16(-acc[0] * b0, -acc[1] * b1);
    *reinterpret_cast<uint32_t*>(TP + sw128_offset(r + 8, n, 128)) =
        pack_bf16(-acc[2] * b0, -acc[3] * b1);
}

// Warps 0..3: output tile (block i = 1 or 3, columns 8nt..8nt+7 of block i-1).
__device__ __forceinline__ void solve_level2(const float* FA, float* FT, float* MS, int warp,
                                             int lane, unsigned char* TP, const float* sbeta) {
    if (warp >= 4) return;
    const int g = lane >> 2, t = lane & 3;
    const int i = (warp >> 1) ? 3 : 1, nt = warp & 1;
    const int r0 = 16 * i, c0 = r0 - 16, n0 = c0 + 8 * nt;
    float* M = MS + warp * 128;  // private 16 x 8
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 2; ks++) {  // M = A_{i,i-1} T_{i-1,i-1}[:, n0..]
        const int k0 = c0 + 8 * ks;
        uint32_t af[4];
        ldsm_a_tf32(FA, LDA, r0, k0, lane, af);
        const uint32_t bf[2] = {to_tf32(FT[(k0 + t) * LDT + n0 + g]),
                                to_tf32(FT[(k0 + t + 4) * LDT + n0 + g])};
        mma_tf32(acc, af, bf);
    }
    *reinterpret_cast<float2*>(M + g * 8 + 2 * t) = make_float2(acc[0], acc[1]);
    *reinterpret_cast<float2*>(M + (g + 8) * 8 + 2 * t) = make_float2(acc[2], acc[3]);
    __syncwarp();
    float out[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < 2; ks++) {  // T_{i,i-1} = -T_ii M
        const int k0 = 8 * ks;
        uint32_t af[4];
        ldsm_a_tf32(FT, LDT, r0, r0 + k0, lane, af);
        const uint32_t bf[2] = {to_tf32(M[(k0 + t) * 8 + g]), to_tf32(M[(k0 + t + 4) * 8 + g])};
        mma_tf32(out, af, bf);
    }
    FT[(r0 + g) * LDT + n0 + 2 * t] = -out[0];
    FT[(r0 + g) * LDT + n0 + 2 * t + 1] = -out[1];
    FT[(r0 + g + 8) * LDT + n0 + 2 * t] = -out[2];
    FT[(r0 + g + 8) * LDT + n0 + 2 * t + 1] = -out[3];
    store_tprime(TP, sbeta, r0 + g, n0 + 2 * t, out);
}

// Warps 0..7: output tile (16-row block 2 + rt, columns 8nt..8nt+7 of 0..31).
// Rows 0..31 of A are dead by now; they hold the private slabs.
__device__ __forceinline__ void solve_level3(float* FA, const float* FT, int warp, int lane,
                                             unsigned char* TP, const float* sbeta) {
    if (warp >= 8) return;
    const int g = lane >> 2, t = lane & 3;
    const int rt = warp >> 2, nt = warp & 3;
    const int n0 = 8 * nt, kb = 2 * (nt >> 1);  // T[k, n0..] = 0 for k < 8 kb
    float* M = FA + warp * 256;                  // private 32 x 8
    static_assert(8 * 256 <= 32 * LDA, "level-3 slabs overlap live rows of A");
#pragma unroll
    for (int mt = 0; mt < 2; mt++) {  // M = A_[23][01] T_[01][01][:, n0..]
        if (mt > rt) break;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const int ra = 32 + 16 * mt;
#pragma unroll
        for (int ks = 0; ks < 4; ks++) {
            if (ks < kb) continue;
            const int k0 = 8 * ks;
            uint32_t af[4];
            ldsm_a_tf32(FA, LDA, ra, k0, lane, af);
            const uint32_t bf[2] = {to_tf32(FT[(k0 + t) * LDT + n0 + g]),
                                    to_tf32(FT[(k0 + t + 4) * LDT + n0 + g])};
            mma_tf32(acc, af, bf);
        }
        float* Mm = M + 16 * mt * 8;
        *reinterpret_cast<float2*>(Mm + g * 8 + 2 * t) = make_float2(acc[0], acc[1]);
        *reinterpret_cast<float2*>(Mm + (g + 8) * 8 + 2 * t) = make_float2(acc[2], acc[3]);
    }
    __syncwarp();
    float out[4] = {0.f, 0.f, 0.f, 0.f};
    const int r0 = 32 + 16 * rt;
#pragma unroll
    for (int ks = 0; ks < 4; ks++) {  // T_[23][01] = -T_[23][23] M
        if (ks >= 2 * (rt + 1)) break;
        const int k0 = 8 * ks;
        uint32_t af[4];
        ldsm_a_tf32(FT, LDT, r0, 32 + k0, lane, af);
        const uint32_t bf[2] = {to_tf32(M[(k0 + t) * 8 + g]), to_tf32(M[(k0 + t + 4) * 8 + g])};
        mma_tf32(out, af, bf);
    }
    store_tprime(TP, sbeta, r0 + g, n0 + 2 * t, out);
}

// SEG: the kernel serves the segment and correction passes (runtime task
// decode); the whole-sequence instantiation compiles without any of it.
// DIO: channels of the caller's q, k, v, g, o, h0, hT and ckpt. 128, or 64
// (whole sequences only), run as d = 128 with channels 64..127 zero: the
// tensor maps fill them with zeros on load and clip them on store, and the
// state's rows and columns past DIO stay exactly zero (k, v = 0 there and the
// decay e^0 = 1 keeps a zero row or column zero), so only the caller's state
// tensors need the stride DIO.
template <bool SEG, int DIO>
__global__ void __launch_bounds__(kThreads, 1)
    kda_chunk_tc_kernel(const __grid_constant__ CUtensorMap map_q,
                        const __grid_constant__ CUtensorMap map_k,
                        const __grid_constant__ CUtensorMap map_v,
                        const __grid_constant__ CUtensorMap map_g,
                        const __grid_constant__ CUtensorMap map_o, const TcParams p) {
    static_assert(DIO == kD || (DIO == 64 && !SEG), "d = 64 runs whole sequences only");
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // Align to 1024 bytes (the 128-byte swizzle atom) by offsetting the
    // __shared__ array itself, so every access below stays an LDS/STS: an
    // integer round trip would turn them into generic loads and stores.
    unsigned char* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    __shared__ uint64_t bars[NBAR];
    __shared__ uint32_t tmem_slot;
    // Runs with v = 0 (transitions, corrections): some lane of the incoming
    // state of the chunk of parity p is nonzero.
    __shared__ int s_nz[2];

    const int tid = threadIdx.x, warp = tid >> 5;
    // TMEM view of a warp: lane quarter q (lanes 32q..32q+31), column group u.
    const int q = warp & 3, u = warp >> 2;
    const int lane = 32 * q + (tid & 31);
    const int T = p.T;
    // Segment and correction passes may be launched as programmatic dependents
    // of the kernel before them: nothing is read before that kernel is done.
    if (SEG) asm volatile("griddepcontrol.wait;" ::: "memory");
    int nseg = p.nseg, seg_chunks = p.seg_chunks, lead = p.lead;
    if (SEG && p.plan) {
        // clamped to the grid and workspace this launch was sized for
        nseg = min(max(__ldg(p.plan), 1), p.nseg);
        seg_chunks = max(__ldg(p.plan + 1), 1);
        lead = max(__ldg(p.plan + 2), 1);
        const long long ntasks = p.pass == 1 ? (long long)p.BH * (2 * nseg - 1)
                                             : (long long)p.BH * (nseg - 1);
        if ((long long)blockIdx.x >= ntasks) return;  // before any barrier or TMEM
    }
    // This CTA's task (see TcParams): kind 0 runs a whole sequence or a segment
    // from h0 / zero writing o, kind 1 a segment from the identity with v = 0
    // (its transition), kind 2 a segment from its incoming state with v = 0,
    // adding to o. Only kind and the first token stay live; the state
    // pointers are formed where they are used.
    const int kind = !SEG                          ? 0
                     : p.pass == 3                 ? 1
                     : p.pass == 2 || p.pass == 4  ? 2
                     : (p.pass == 1 && (int)blockIdx.x >= p.BH * nseg) ? 1
                                                                          : 0;
    const bool v_zero = kind != 0;
    const bool whole = !SEG || p.pass == 0 || p.pass >= 3;  // one CTA runs all the chunks
    auto task_seq = [&](int* bh_out, int* seg_out) {
        int bh = blockIdx.x, seg = 0;
        if (whole) {
        } else if (kind == 2 || kind == 1) {
            const int j = kind == 1 ? (int)blockIdx.x - p.BH * nseg : (int)blockIdx.x;
            bh = j / (nseg - 1);
            seg = 1 + j % (nseg - 1);
        } else if (SEG && p.pass == 1 && (int)blockIdx.x >= p.BH) {
            const int j = (int)blockIdx.x - p.BH;
            bh = j / (nseg - 1);
            seg = 1 + j % (nseg - 1);
        }
        *bh_out = bh;
        *seg_out = seg;
    };
    int bh, seg;
    task_seq(&bh, &seg);
    int b = bh / p.H, h = bh % p.H;
    int t_begin = seg == 0 ? 0 : (lead + seg - 1) * seg_chunks * kC;
    // Initial state: h0 (whole sequences and first segments), zero (other
    // segments), the identity (transition runs) or the incoming state.
    const float* h0p = (kind == 2 && whole) ? p.ws_sin + (size_t)bh * kD * kD
                       : kind == 2 ? p.ws_sin + ((size_t)bh * (nseg - 1) + seg - 1) * kD * kD
                       : (kind == 0 && seg == 0 && p.h0) ? p.h0 + (size_t)bh * DIO * DIO
                                                         : nullptr;
    int nchunks = whole
                      ? (T + kC - 1) / kC
                      : min(seg == 0 ? lead * seg_chunks : seg_chunks,
                            (T - t_begin + kC - 1) / kC);
    // Tasks of this CTA: one, except in the balanced schedule, where the range
    // [lo, hi) of chunk steps gives the head of sequence s_last (chunks
    // [0, c_last), when c_last < nch), the whole sequences between, and the
    // tail of sequence s_first (chunks [c_first, nch), when c_first > 0).
    const bool bal = !SEG && p.bal_W > 0;
    const int nch = (T + kC - 1) / kC;
    int ntask = 1, s_first = 0, c_first = 0, s_last = 0, c_last = 0, full_lo = 0;
    bool has_head = false, has_tail = false;
    if (bal) {
        const long long lo = (long long)blockIdx.x * p.bal_W;
        const long long hi = min(lo + p.bal_W, (long long)p.BH * nch);
        ntask = 0;
        if (lo < hi) {
            s_first = (int)(lo / nch);
            c_first = (int)(lo % nch);
            s_last = (int)((hi - 1) / nch);
            c_last = (int)((hi - 1) % nch) + 1;
            has_tail = c_first > 0;
            has_head = c_last < nch;
            full_lo = has_tail ? s_first + 1 : s_first;
            const int full_hi = has_head ? s_last - 1 : s_last;
            ntask = (has_head ? 1 : 0) + max(0, full_hi - full_lo + 1) + (has_tail ? 1 : 0);
        }
    }
    bool from_slot = false, to_slot = false;
    auto set_task = [&](int ti) {  // balanced schedule: task ti in run order
        int c0 = 0, c1 = nch;
        from_slot = to_slot = false;
        if (has_head && ti == 0) {
            bh = s_last;
            c1 = c_last;
            to_slot = true;
        } else if (has_tail && ti == ntask - 1) {
            bh = s_first;
            c0 = c_first;
            from_slot = true;
        } else {
            bh = full_lo + ti - (has_head ? 1 : 0);
        }
        b = bh / p.H;
        h = bh % p.H;
        t_begin = c0 * kC;
        nchunks = c1 - c0;
        h0p = from_slot ? p.bal_states + (size_t)bh * kD * kD
              : p.h0    ? p.h0 + (size_t)bh * DIO * DIO
                        : nullptr;
    };
    if (bal && ntask > 0) set_task(0);
    const uint32_t sbase = smem_addr(sm);
    float* sbeta = reinterpret_cast<float*>(sm + OFF_BETA);
    float* slam = reinterpret_cast<float*>(sm + OFF_LAM);
    int flags = 0;
    bool failed = false, zero_exit = false;

    if (tid == 0) {
        s_nz[0] = s_nz[1] = 0;
        for (int i = 0; i < NBAR; i++)
            mbar_init(&bars[i], (i == BAR_P1 || i == BAR_GP) ? kThreads : 1);
        fence_mbarrier_init();
        if (nchunks > 0) {
            prefetch_tensormap(&map_q);
            prefetch_tensormap(&map_k);
            prefetch_tensormap(&map_v);
            prefetch_tensormap(&map_g);
        }
    }
    if (warp == 0) {
        tmem_alloc(&tmem_slot, TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_slot;
    const uint32_t tq = tmem_at(tbase, 32 * q, 0);  // this warp's lane quarter

    auto issue_qk = [&](int c) {
        mbar_arrive_expect_tx(&bars[BAR_QK], 4 * 8192);
        const int t0 = t_begin + c * kC;
        tma_load_4d(sm + OFF_KQP, &map_k, &bars[BAR_QK], 0, h, t0, b);
        tma_load_4d(sm + OFF_KQP + 16384, &map_k, &bars[BAR_QK], 64, h, t0, b);
        tma_load_4d(sm + OFF_KQP + 8192, &map_q, &bars[BAR_QK], 0, h, t0, b);
        tma_load_4d(sm + OFF_KQP + 16384 + 8192, &map_q, &bars[BAR_QK], 64, h, t0, b);
    };
    auto issue_g = [&](int c) {
        mbar_arrive_expect_tx(&bars[BAR_G], 32768);
#pragma unroll
        for (int cbk = 0; cbk < 4; cbk++)
            tma_load_4d(sm + OFF_G + cbk * 8192, &map_g, &bars[BAR_G], 32 * cbk, h, t_begin + c * kC,
                        b);
    };
    auto issue_v = [&](int c) {
        mbar_arrive_expect_tx(&bars[BAR_V], 2 * 8192);
        tma_load_4d(sm + OFF_V, &map_v, &bars[BAR_V], 0, h, t_begin + c * kC, b);
        tma_load_4d(sm + OFF_V + 8192, &map_v, &bars[BAR_V], 64, h, t_begin + c * kC, b);
    };
    // beta is strided by H in memory: plain loads, kept one chunk ahead.
    auto load_beta = [&](int c) {
        const int t = t_begin + c * kC + tid;
        return (tid < kC && c < nchunks && t < T) ? p.beta[((size_t)b * T + t) * p.H + h] : 0.f;
    };
    float beta_next = 0.f;

    // T' is zero in the six 16 x 16 blocks above the diagonal; nothing else
    // writes there, so they are cleared once.
    for (int e = tid; e < 6 * 128; e += kThreads) {
        const int blkid = e >> 7, i = (e >> 3) & 15, jp = e & 7;
        const int br = blkid < 3 ? 0 : (blkid < 5 ? 1 : 2);
        const int bc = blkid < 3 ? blkid + 1 : (blkid < 5 ? blkid - 1 : 3);
        *reinterpret_cast<uint32_t*>(sm + OFF_A0 + sw128_offset(16 * br + i, 16 * bc + 2 * jp, 128)) =
            0u;
    }
    // The 64 x 64 identity that copies the v tile into D1 (V^T x I).
    for (int e = tid; e < 64 * 32; e += kThreads) {
        const int r = e >> 5, cp = 2 * (e & 31);
        const uint32_t w = (r == cp ? 0x3F80u : 0u) | (r == cp + 1 ? 0x3F800000u : 0u);
        *reinterpret_cast<uint32_t*>(sm + OFF_I + sw128_offset(r, cp, 64)) = w;
    }
    // Likewise P's upper right 32 x 32 block (rows 0..31, columns 32..63).
    for (int e = tid; e < 32 * 16; e += kThreads)
        *reinterpret_cast<uint32_t*>(sm + OFF_A0 + sw128_offset(64 + (e >> 4), 32 + 2 * (e & 15), 128)) = 0u;
    // O of chunk cc -> global: O^T sits in D1 columns 64 + r (token r), lane j
    // (value channel j); warp column group u takes tokens [16u, 16u + 16), so a
    // warp store covers 32 consecutive value channels of one token.
    auto write_o = [&](int cc, int len, const float* x) {
        // A NaN or Inf in q, k or v reaches some output through the
        // recurrence; x * 0 is 0 for finite x and NaN otherwise.
        float pr[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int e = 0; e < 16; e++) pr[e & 3] = fmaf(x[e], 0.f, pr[e & 3]);
        if ((pr[0] + pr[1]) + (pr[2] + pr[3]) != 0.f) flags |= KDA_DEV_NONFINITE;
        if (kind == 0) {  // staged: one TMA store writes the chunk's rows (rows past T are clipped)
            __nv_bfloat16* st = reinterpret_cast<__nv_bfloat16*>(sm + OFF_OST) + 16 * u * kD + lane;
#pragma unroll
            for (int e = 0; e < 16; e++) st[e * kD] = __float2bfloat16_rn(x[e]);
            return;
        }
        __nv_bfloat16* dst = p.o + (((size_t)b * T + t_begin + cc * kC) * p.H + h) * kD + lane;
        const size_t rs = (size_t)p.H * kD;
#pragma unroll
        for (int e = 0; e < 16; e++) {
            const int r = 16 * u + e;
            if (r < len) {
                float val = x[e];
                if (kind == 2) val += __bfloat162float(dst[r * rs]);  // o += this pass's part
                dst[r * rs] = __float2bfloat16_rn(val);
            }
        }
    };
    auto store_o = [&](int cc, int len) {
        if (kind == 1) return;
        float x[16];
        tmem_ld16(tq + TM_D1 + 64 + 16 * u, x);
        write_o(cc, len, x);
    };

    uint32_t mma_phase = 0;
    auto mma_wait = [&]() {
        bool ok = mbar_wait(&bars[BAR_MMA], mma_phase);
        mma_phase ^= 1u;
        return ok;
    };
    // Round 4 completes on its own barrier and is waited for only when its
    // results (S, the O rows, the U and Kb operands' buffers) are next needed,
    // so the following chunk's decay scan and operand build run under it.
    uint32_t r4_phase = 0, r2_phase = 0;
    bool r4_pending = false;
    auto r4_wait = [&]() {
        bool ok = true;
        if (r4_pending) {
            ok = mbar_wait(&bars[BAR_R4], r4_phase);
            r4_phase ^= 1u;
            r4_pending = false;
        }
        tc_fence_after();
        return ok;
    };

    // Chunks this CTA has run in earlier tasks: the per-chunk mbarriers
    // complete once per chunk, so their phase is the parity of the running
    // chunk count.
    int gc = 0;
    for (int ti = 0; ti < ntask && !failed; ti++) {
    if (bal && ti > 0) set_task(ti);
    if (tid == 0 && nchunks > 0) {
        issue_qk(0);
        issue_g(0);
        if (!v_zero) issue_v(0);
    }
    beta_next = load_beta(0);
    if (from_slot) {
        // The head of this sequence ran first on the previous CTA; its final
        // state is in the slot once the flag is set. The wait is bounded by
        // far more than a head can take (at most nch chunks, ~5 us each).
        bool waited = true;
        if (tid == 0) {
            const long long t0 = clock64(), limit = max(1LL << 31, (long long)nch << 22);
            while (ld_acquire_gpu(p.bal_flags + bh) == 0) {
                if (clock64() - t0 > limit) { waited = false; break; }
            }
        }
        if (__syncthreads_or(!waited)) { failed = true; break; }
    }
    // Incoming state -> TMEM, transposed: lane j = value channel j, column i
    // = key channel i (a warp reads 128 contiguous bytes of a state row per load).
    {
        float x[32];
#pragma unroll
        for (int e = 0; e < 32; e++) {
            const int i = 32 * u + e;
            x[e] = kind == 1 ? (lane == i ? 1.f : 0.f)
                   : from_slot ? __ldcg(h0p + (size_t)i * kD + lane)
                   : (h0p && (DIO == kD || (i < DIO && lane < DIO)) ? h0p[(size_t)i * DIO + lane] : 0.f);
        }
        tmem_st16(tq + TM_S + 32 * u, x);
        tmem_st16(tq + TM_S + 32 * u + 16, x + 16);
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    for (int c = 0; c < nchunks && !failed; c++) {
        const uint32_t par = (uint32_t)((gc + c) & 1);

        // ------------------------------------------------------------ P1
        // Warp w owns channels 8w .. 8w + 7 of all four tiles; lane (a, j) =
        // (lane / 8, lane % 8) owns rows 16a + j and 16a + j + 8 (so the 32
        // lanes' row addresses cover all eight swizzle positions). Tile
        // totals and decay constants never leave the warp: they go through
        // the warp's own rows of the g buffer once its g values are read.
        // Log-decays are kept in log2 units: each exponential is one ex2.
        bool ok = mbar_wait(&bars[BAR_QK], par) && mbar_wait(&bars[BAR_G], par);
        if (!ok) flags |= KDA_DEV_TIMEOUT;  // voted on after the Gram readout
        {
            const int ln = tid & 31;
            const int a = ln >> 3, j = ln & 7;
            const int c0 = 8 * warp;
            // this warp's 8 channels in the g buffer: block c0 / 32, chunks
            // 2 (w % 4) and 2 (w % 4) + 1 of each 128-byte row (swizzled)
            unsigned char* gblk = sm + OFF_G + (c0 >> 5) * 8192;
            const uint32_t gch = 2u * (uint32_t)(warp & 3);
            auto grow_chunk = [&](int r, int half) {
                return gblk + r * 128 + (((gch + (uint32_t)half) ^ (uint32_t)(r & 7)) << 4);
            };
            if (tid < kC) {
                flags |= finite_flag(beta_next);
                sbeta[tid] = beta_next;
            }
            beta_next = load_beta(c + 1);
            float cv6[5];
            // Decay scan, one column per lane: lane (a, j) takes channel c0 + j
            // of tile a, its 16 rows in the order 2a, 2a + 1, .. (mod 16), so the
            // rows one load touches lie in four different swizzle classes.
            // Rows i and i + 8 of the order share a class and differ in byte
            // offset by 1024.
            {
                const uint32_t cb = gch + (uint32_t)(j >> 2), w4 = 4u * (uint32_t)(j & 3);
                uint32_t off[8];
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    const uint32_t rr = (uint32_t)((i + 2 * a) & 15);
                    off[i] = (uint32_t)(16 * a + rr) * 128u + ((cb ^ (rr & 7u)) << 4) + w4;
                }
                float sc[16];  // inclusive sums along the rotated order, log2 units
                float mn = 0.f, mx = -5.f, run = 0.f;
#pragma unroll
                for (int i = 0; i < 16; i++) {
                    const float x = *reinterpret_cast<const float*>(gblk + (off[i & 7] ^ (i >= 8 ? 1024u : 0u)));
                    mn = fminf(mn, x);
                    mx = fmaxf(mx, x);
                    run = fmaf(x, kLog2e, run);
                    sc[i] = run;
                }
                const float tot = sc[15];
                if (!(fabsf(tot) <= 3.402823466e38f)) flags |= KDA_DEV_NONFINITE;
                else if (mn < kLogDecayMin || mx > 0.f) flags |= KDA_DEV_DECAY_RANGE;
                // rows 2a .. 15 come first in the order: natural prefix =
                // sc + (rows 0 .. 2a - 1) there, sc - (rows 2a .. 15) after the wrap
                const float tail = a == 0 ? sc[15] : a == 1 ? sc[13] : a == 2 ? sc[11] : sc[9];
                const float head = tot - tail;
#pragma unroll
                for (int i = 0; i < 16; i++) {
                    const float pv = (2 * a <= 15 - i) ? sc[i] + head : sc[i] - tail;
                    *reinterpret_cast<float*>(gblk + (off[i & 7] ^ (i >= 8 ? 1024u : 0u))) = pv;
                }
                // Per (tile, channel) decay constants of tile a, channel c0 + j:
                //   0: e^{G_a-}  1: e^{G_C - G_a+}  2: e^{tile total}  4, 5: e^{G_{a'-} - G_a+}, a' = 2, 3
                // (a' = 1 would be e^0 for tile 0: not stored)
                float tb[4];
#pragma unroll
                for (int bb = 0; bb < 4; bb++) tb[bb] = __shfl_sync(0xffffffffu, tot, 8 * bb + j);
                float pre = 0.f, post = 0.f;
#pragma unroll
                for (int bb = 0; bb < 4; bb++) {
                    if (bb < a) pre += tb[bb];
                    if (bb > a) post += tb[bb];
                }
                cv6[0] = fast_exp2(pre);
                cv6[1] = fast_exp2(post);
                cv6[2] = fast_exp2(tot);
                cv6[3] = fast_exp2(a < 1 ? tb[1] : 0.f);
                cv6[4] = fast_exp2((a < 1 ? tb[1] : 0.f) + (a < 2 ? tb[2] : 0.f));
                if (a == 0) slam[c0 + j] = fast_exp2(tb[0] + tb[1] + tb[2] + tb[3]);
            }
            __syncwarp();  // the column prefixes are in the g buffer
            float gam[2][8];  // in-tile inclusive cumulative log2-decay, rows j and j + 8
#pragma unroll
            for (int e = 0; e < 2; e++) {
                const int r = 16 * a + j + 8 * e;
#pragma unroll
                for (int hq = 0; hq < 2; hq++) {
                    const float4 v = *reinterpret_cast<const float4*>(grow_chunk(r, hq));
                    gam[e][4 * hq] = v.x; gam[e][4 * hq + 1] = v.y;
                    gam[e][4 * hq + 2] = v.z; gam[e][4 * hq + 3] = v.w;
                }
            }
            __syncwarp();  // every lane has its prefixes: rows 0 .. 19 take the constants
#pragma unroll
            for (int k5 = 0; k5 < 5; k5++)
                reinterpret_cast<float*>(grow_chunk(5 * a + k5, j >> 2))[j & 3] = cv6[k5];
            __syncwarp();
            float cst[6][8];
#pragma unroll
            for (int k6 = 0; k6 < 6; k6++) {
                if (k6 == 3) {
#pragma unroll
                    for (int z = 0; z < 8; z++) cst[3][z] = 1.f;
                    continue;
                }
                const int k5 = k6 < 3 ? k6 : k6 - 1;
                const float4 w0 = *reinterpret_cast<const float4*>(grow_chunk(5 * a + k5, 0));
                const float4 w1 = *reinterpret_cast<const float4*>(grow_chunk(5 * a + k5, 1));
                cst[k6][0] = w0.x; cst[k6][1] = w0.y; cst[k6][2] = w0.z; cst[k6][3] = w0.w;
                cst[k6][4] = w1.x; cst[k6][5] = w1.y; cst[k6][6] = w1.z; cst[k6][7] = w1.w;
            }
            const uint32_t blk = (uint32_t)(c0 >> 6);
            const uint32_t chunk = (uint32_t)((c0 & 63) >> 3);
#pragma unroll
            for (int e = 0; e < 2; e++) {
                const int r = 16 * a + j + 8 * e;
                const uint32_t ro = (uint32_t)r * 128u + ((chunk ^ (uint32_t)(r & 7)) << 4);
                unsigned char* pk = sm + OFF_KQP + blk * 16384u + ro;
                unsigned char* pq = pk + 8192u;
                float kf[8], qf[8], e1[8], em[8];
                unpack8(*reinterpret_cast<const uint4*>(pk), kf);
                unpack8(*reinterpret_cast<const uint4*>(pq), qf);
#pragma unroll
                for (int z = 0; z < 8; z++) {
                    e1[z] = fast_exp2(gam[e][z]);   // e^{G_r - G_a-} <= 1
                    em[z] = fast_exp2(-gam[e][z]);  // e^{G_a- - G_r} < e^80
                }
                float kp[8], qp[8], ke[8], t8[8];
#pragma unroll
                for (int z = 0; z < 8; z++) {
                    kp[z] = kf[z] * e1[z];
                    qp[z] = qf[z] * e1[z];
                    t8[z] = kf[z] * em[z];                // own window: bounded reciprocal decay
                    ke[z] = t8[z] * cst[2][z];            // k e^{G_a+ - G_r}, <= |k|
                }
                *reinterpret_cast<uint4*>(pk) = pack8(kp);
                *reinterpret_cast<uint4*>(pq) = pack8(qp);
                unsigned char* pw = sm + OFF_KM + blk * (KM_ROWS * 128u) + ro;
                *reinterpret_cast<uint4*>(pw + (uint32_t)win_row(a) * 128u) = pack8(t8);
#pragma unroll
                for (int ap = 1; ap < 4; ap++) {
                    if (ap > a) {
#pragma unroll
                        for (int z = 0; z < 8; z++) t8[z] = ke[z] * cst[2 + ap][z];
                        *reinterpret_cast<uint4*>(pw + (uint32_t)win_row(ap) * 128u) = pack8(t8);
                    }
                }
                // Kt, Qt (round 2 of the previous chunk has read its copies) and
                // Kb (into this chunk's parity buffer: round 4 of the previous
                // chunk may still read the other).
#pragma unroll
                for (int z = 0; z < 8; z++) t8[z] = -(kp[z] * cst[0][z]);  // -Kt: round 2 subtracts Y
                *reinterpret_cast<uint4*>(sm + OFF_AKQ + 2 * blk * 8192u + ro) = pack8(t8);
#pragma unroll
                for (int z = 0; z < 8; z++) t8[z] = qp[z] * cst[0][z];
                *reinterpret_cast<uint4*>(sm + OFF_AKQ + 2 * blk * 8192u + 8192 + ro) = pack8(t8);
#pragma unroll
                for (int z = 0; z < 8; z++) t8[z] = ke[z] * cst[1][z];
                *reinterpret_cast<uint4*>(sm + (par ? OFF_KB1 : OFF_KB) + blk * 8192u + ro) =
                    pack8(t8);
            }
        }
        // Only the Gram MMA and the next g load need every warp's operands
        // and reads done: the other warps go on to their stores at once.
        fence_proxy_async_smem();
        mbar_arrive(&bars[BAR_P1]);

        // ------------------------------------------------------------ round 1: Gram
        if (tid == kIssueThread) {
            if (!mbar_wait(&bars[BAR_P1], par)) flags |= KDA_DEV_TIMEOUT;
            tc_fence_after();
            // The four windows are consecutive rows of one tile, so a single
            // N = 160 product computes every Gram block: columns win_row(a)..
            // of D hold the block anchored at tile a.
            const uint64_t ad0 = desc_kmajor(sbase + OFF_KQP);
            const uint64_t bd0 = desc_kmajor(sbase + OFF_KM);
            const uint32_t idesc = idesc_bf16(128, KM_ROWS, 0, 0);
#pragma unroll
            for (int kk = 0; kk < 8; kk++)
                mma_bf16(tbase + TM_SCR, ad0 + kstep_kmajor(128, kk), bd0 + kstep_kmajor(KM_ROWS, kk),
                         idesc, kk > 0);
            mma_commit(&bars[BAR_MMA]);
            if (c + 1 < nchunks) issue_g(c + 1);  // every warp is done with the g buffer
        }
        // Kb, U (under [Kt; Qt]), D1 and S are free again. (A timeout flag is
        // only ever set by a failed wait, so it fails the vote after the readout.)
        ok = r4_wait() && !(flags & KDA_DEV_TIMEOUT);
        if (!ok) flags |= KDA_DEV_TIMEOUT;
        // The O staging buffer: the previous chunk's store has read it (its
        // issuer arrived on BAR_P1 after waiting for that).
        if (kind == 0 && !mbar_wait(&bars[BAR_P1], par)) flags |= KDA_DEV_TIMEOUT;
        if (ok) {
            // The previous (full) chunk's O rows (D1 columns 64..127) -> global;
            // S0^T (lane = value channel, columns = key channels 32u ..) -> bf16
            // A operand of round 2 in TMEM; S <- e^{G_C} S (per key channel).
            float y[32];
            if (c > 0 && kind != 1) {
                float xo[16];
                tmem_ld16_32(tq + TM_D1 + 64 + 16 * u, tq + TM_S + 32 * u, xo, y);
                write_o(c - 1, kC, xo);
            } else {
                tmem_ld32(tq + TM_S + 32 * u, y);
            }
            {  // round 2 accumulates onto D1: (Qt S0)^T starts from zero
                float zz[16];
#pragma unroll
                for (int e = 0; e < 16; e++) zz[e] = 0.f;
                tmem_st16(tq + TM_D1 + 64 + 16 * u, zz);
            }
            if (SEG && v_zero) {
                bool nz = false;
#pragma unroll
                for (int e = 0; e < 32; e++) nz = nz || (y[e] != 0.f);  // NaN counts as nonzero
                if (__any_sync(0xffffffffu, nz) && (tid & 31) == 0) s_nz[par] = 1;
            }
            {
                float pk[16];
#pragma unroll
                for (int e = 0; e < 16; e++) pk[e] = pack2f(y[2 * e], y[2 * e + 1]);
                tmem_st16(tq + TM_AUX + 16 * u, pk);
            }
            // e^{G_C} of these key channels comes from other warps' decay
            // constants, as does the beta the readout uses: every warp has
            // arrived on BAR_P1 after writing them.
            if (!mbar_wait(&bars[BAR_P1], par)) flags |= KDA_DEV_TIMEOUT;
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                const float4 l4 = *reinterpret_cast<const float4*>(slam + 32 * u + e);
                y[e] *= l4.x; y[e + 1] *= l4.y; y[e + 2] *= l4.z; y[e + 3] *= l4.w;
            }
            tmem_st16(tq + TM_S + 32 * u, y);
            tmem_st16(tq + TM_S + 32 * u + 16, y + 16);
            tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars[BAR_GP]);  // stash stores in shared memory, S0^T copy in TMEM
        ok = mma_wait() && ok;
        tc_fence_after();
        // Each warp waited for the Gram round itself; the next q, k tiles may
        // land as soon as it is done. A failure is voted on after the readout.
        if (tid == kTmaThread && c + 1 < nchunks) issue_qk(c + 1);

        // Gram readout. Quarter q: rows 32(q&1).. of A (q < 2) or P (q >= 2);
        // warp u writes output columns [16u, 16u + 16). Only blocks that are
        // read are written: the solve reads A strictly below the diagonal (its
        // diagonal blocks' upper parts are loaded but never used), and P's
        // blocks right of the diagonal are zero (the upper right 32 x 32 block
        // is cleared once; warps u > a0 + 1 have nothing to write).
        auto readout = [&](int ug) {  // column group ug of this warp's lane quarter
            const int part = q >> 1;
            const int r = 32 * (q & 1) + (tid & 31);
            const int a = r >> 4, a0 = 2 * (q & 1);
            if (ug <= a0 + 1) {
                float v0[16], v1[16];
                if (ug <= a0) {
                    tmem_ld16x2(tq + TM_SCR + win_row(a0) + 16 * ug, tq + TM_SCR + win_row(a0 + 1) + 16 * ug,
                                v0, v1);
                } else {
                    tmem_ld16(tq + TM_SCR + win_row(a0 + 1) + 16 * ug, v1);
#pragma unroll
                    for (int jj = 0; jj < 16; jj++) v0[jj] = v1[jj];  // rows of tile a0: not read
                }
                const bool second = (a == a0 + 1);
                float out[16];
                if (part == 0) {
                    const float br = sbeta[r];
#pragma unroll
                    for (int jj = 0; jj < 16; jj++) out[jj] = br * (second ? v1[jj] : v0[jj]);
                    float4* FA = reinterpret_cast<float4*>(sm + OFF_FA + (r * LDA + 16 * ug) * 4);
#pragma unroll
                    for (int jj = 0; jj < 4; jj++)
                        FA[jj] = make_float4(out[4 * jj], out[4 * jj + 1], out[4 * jj + 2], out[4 * jj + 3]);
                } else {
#pragma unroll
                    for (int jj = 0; jj < 16; jj++) {
                        const int s = 16 * ug + jj;
                        const float val = second ? v1[jj] : v0[jj];
                        out[jj] = (ug < a || (ug == a && s <= r)) ? val : 0.f;
                    }
                    st_row8(sm + OFF_A0, 64 + r, 16 * ug, 128, out);
                    st_row8(sm + OFF_A0, 64 + r, 16 * ug + 8, 128, out + 8);
                }
            }
        };
        // A rows by their own column group; P rows, read only by round 4, by
        // warps 10, 11, 14, 15 (idle until round 2) so that the solve warps
        // 2, 3, 6, 7 leave the readout at once.
        if (q < 2) {
            readout(u);
        } else if (u >= 2) {
            if (q == 2) {
                readout(u - 2);
            } else {
                readout(2 * (u - 2));
                readout(2 * (u - 2) + 1);
            }
        }
        tc_fence_before();
        if (SEG && v_zero) {  // runs with v = 0 decide on an early stop here: a CTA barrier
            if (__syncthreads_or(!ok)) { failed = true; break; }
        } else {
            if (!ok) flags |= KDA_DEV_TIMEOUT;  // voted on at the end of the solve
            // Each diagonal block's warp waits for the warp that wrote its A rows
            // (block 0: itself; 1: warp 4; 2: warp 9, which also wrote A_32; 3:
            // warp 13). A_10 is warp 0's, A_[23][01] that of warps 1 and 5,
            // which reach the level-3 barrier after writing it.
            if (warp == 1 || warp == 4) named_sync(5, 64);
            else if (warp == 2 || warp == 9) named_sync(6, 64);
            else if (warp == 3 || warp == 13) named_sync(7, 64);
        }
        if (!SEG || !(v_zero && s_nz[par] == 0)) {
            if (tid == kR2Thread) {
                // Round 2: D1 = [Kt; Qt] S0 = [Y; Qt S0], under the solve.
                if (!mbar_wait(&bars[BAR_GP], par)) flags |= KDA_DEV_TIMEOUT;
                tc_fence_after();
                // D1[:, 0:64] = V^T (V^T x I; A = the v tile, MN-major), then
                // D1^T += S0^T [-Kt; Qt]^T: [(V - Y)^T | (Qt S0)^T], A = S0^T in TMEM.
                if (!v_zero) {
                    if (!mbar_wait(&bars[BAR_V], par)) flags |= KDA_DEV_TIMEOUT;
                    tc_fence_after();
                    const uint32_t idesc_v = idesc_bf16(128, 64, 1, 0);
                    const uint64_t vd0 = desc_mnmajor(sbase + OFF_V, 64);
                    const uint64_t id0 = desc_kmajor(sbase + OFF_I);
#pragma unroll
                    for (int kk = 0; kk < 4; kk++)
                        mma_bf16(tbase + TM_D1, vd0 + kstep_mnmajor(kk), id0 + kstep_kmajor(64, kk),
                                 idesc_v, kk > 0);
                }
                const uint32_t idesc = idesc_bf16(128, 128, 0, 0);
                const uint64_t bd0 = desc_kmajor(sbase + OFF_AKQ);
#pragma unroll
                for (int kk = 0; kk < 8; kk++)
                    mma_bf16_ta(tbase + TM_D1, tbase + TM_AUX + 8 * kk, bd0 + kstep_kmajor(128, kk),
                                idesc, (!v_zero) || kk > 0);
                mma_commit(&bars[BAR_R2]);
                if (c > 0 && kind == 0) {
                    tma_store_4d(&map_o, sm + OFF_OST, 0, h, t_begin + (c - 1) * kC, b);
                    bulk_wait_read();
                }
            }
        }
        if (SEG && v_zero && s_nz[par] == 0) {
            // With v = 0 and an incoming state that is exactly zero in fp32,
            // every later state and output of the run is exactly zero: the
            // transition is zero and nothing more is added to o. The run
            // stops here, once the tiles already requested have landed.
            zero_exit = true;
            if (tid == 0 && c + 1 < nchunks) {
                const uint32_t np = (uint32_t)((c + 1) & 1);
                if (!mbar_wait(&bars[BAR_QK], np) || !mbar_wait(&bars[BAR_G], np))
                    flags |= KDA_DEV_TIMEOUT;
            }
            break;
        }

        // ------------------------------------------------------------ T = (I + A)^-1
        {
            float* FA = reinterpret_cast<float*>(sm + OFF_FA);
            float* FT = reinterpret_cast<float*>(sm + OFF_FT);
            float* MS = reinterpret_cast<float*>(sm + OFF_MS);
            unsigned char* TP = sm + OFF_A0;  // T' rows 0..63
            if (warp < 4) {  // diagonal 16x16 blocks: warp = block, lane j = column j
                const int o0 = 16 * warp, jc = tid & 15;
                float acc[16], x[16];
#pragma unroll
                for (int i = 0; i < 16; i++) acc[i] = 0.f;
#pragma unroll
                for (int m0 = 0; m0 < 16; m0 += 4) {  // right-looking, four columns of A per load
                    float4 arow[16];
#pragma unroll
                    for (int i = m0 + 1; i < 16; i++)
                        arow[i] = *reinterpret_cast<const float4*>(FA + (o0 + i) * LDA + o0 + m0);
#pragma unroll
                    for (int mm = 0; mm < 4; mm++) {  // finish x_m, push into later rows
                        const int m = m0 + mm;
                        x[m] = (m < jc) ? 0.f : ((m == jc) ? 1.f : -acc[m]);
#pragma unroll
                        for (int i = m + 1; i < 16; i++) {
                            const float am = mm == 0 ? arow[i].x : mm == 1 ? arow[i].y
                                           : mm == 2 ? arow[i].z : arow[i].w;
                            acc[i] += am * x[m];
                        }
                    }
                }
                if ((tid & 31) < 16) {
                    const float bj = sbeta[o0 + jc];
#pragma unroll
                    for (int i = 0; i < 16; i++) {
                        FT[(o0 + i) * LDT + o0 + jc] = x[i];
                        *reinterpret_cast<__nv_bfloat16*>(TP + sw128_offset(o0 + i, o0 + jc, 128)) =
                            __float2bfloat16_rn(x[i] * bj);
                    }
                }
            }
            // Level 2 (warps 0-3) needs only the diagonal blocks of warps 0-3,
            // level 3 (warps 0-7) those and level 2 (its scratch slabs also
            // overwrite rows of A that level 2 reads). The V - Y warps need
            // neither and start as soon as round 2 is done.
            if (warp < 4) named_sync(1, 128);
            solve_level2(FA, FT, MS, warp, tid & 31, TP, sbeta);
            if (warp < 8) named_sync(2, 256);
            solve_level3(FA, FT, warp, tid & 31, TP, sbeta);
            if (warp >= 8) {
                // (V - Y)^T (D1 columns 0..63: tokens) -> bf16 A operand of round 3
                // in TMEM (AUX columns 0..31; S0^T there is consumed), tokens
                // [32 (u - 2), + 32), by the eight warps idle in this level.
                ok = v_zero || mbar_wait(&bars[BAR_V], par);
                ok = mbar_wait(&bars[BAR_R2], r2_phase) && ok;
                tc_fence_after();
                if (ok) {
                    const int t0 = 32 * (u - 2);
                    float y[32], pk[16];
                    tmem_ld32(tq + TM_D1 + t0, y);
#pragma unroll
                    for (int e = 0; e < 16; e++) pk[e] = pack2f(y[2 * e], y[2 * e + 1]);
                    tmem_st16(tq + TM_AUX + t0 / 2, pk);
                    tmem_wait_st();
                }
            }
            r2_phase ^= 1u;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(!ok || (flags & KDA_DEV_TIMEOUT))) { failed = true; break; }
        if (SEG && tid == 0) s_nz[par] = 0;  // every thread has read it

        // ------------------------------------------------------------ round 3: U^T = (V - Y)^T T'^T
        if (tid == 0) {
            tc_fence_after();
            const uint32_t idesc_y = idesc_bf16(128, 64, 0, 0);  // A = (V - Y)^T (TMEM)
            const uint64_t td0 = desc_kmajor(sbase + OFF_A0);    // T': rows 0..63 of [T'; P]
#pragma unroll
            for (int kk = 0; kk < 4; kk++)
                mma_bf16_ta(tbase + TM_D1, tbase + TM_AUX + 8 * kk, td0 + kstep_kmajor(128, kk),
                            idesc_y, kk > 0);
            mma_commit(&bars[BAR_MMA]);
        }
        ok = mma_wait();
        tc_fence_after();
        if (tid == kTmaThread && c + 1 < nchunks && !v_zero) issue_v(c + 1);
        {  // U^T (D1 columns 16u .. + 16: tokens) -> bf16 A operand of round 4 in TMEM
            float x[16], pk[8];
            tmem_ld16(tq + TM_D1 + 16 * u, x);
#pragma unroll
            for (int e = 0; e < 8; e++) pk[e] = pack2f(x[2 * e], x[2 * e + 1]);
            tmem_st8(tq + TM_AUX + 32 + 8 * u, pk);
            tmem_wait_st();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        if (__syncthreads_or(!ok)) { failed = true; break; }

        // ------------------------------------------------------------ round 4: S += Kb^T U, O += P U
        if (tid == kIssueThread) {
            tc_fence_after();
            // S^T += U^T Kb (B = Kb, MN-major), O^T += U^T P^T (B = P, K-major); A = U^T in TMEM
            const uint32_t idesc = idesc_bf16(128, 128, 0, 1);
            const uint64_t kb0 = desc_mnmajor(sbase + (par ? OFF_KB1 : OFF_KB), 64);
#pragma unroll
            for (int kk = 0; kk < 4; kk++)
                mma_bf16_ta(tbase + TM_S, tbase + TM_AUX + 32 + 8 * kk, kb0 + kstep_mnmajor(kk), idesc,
                            1);
            const uint32_t idesc_o = idesc_bf16(128, 64, 0, 0);
            const uint64_t pd0 = desc_kmajor(sbase + OFF_A0 + 64 * 128);  // P: rows 64..127
#pragma unroll
            for (int kk = 0; kk < 4; kk++)
                mma_bf16_ta(tbase + TM_D1 + 64, tbase + TM_AUX + 32 + 8 * kk,
                            pd0 + kstep_kmajor(128, kk), idesc_o, 1);
            mma_commit(&bars[BAR_R4]);
        }
        r4_pending = true;
        // Sparse state checkpoint: only full chunks count, so the slot index
        // stays below n_ckpt = T / ckpt_every.
        if (p.ckpt && (c + 1) % p.ck_chunks == 0 && (c + 1) / p.ck_chunks <= p.n_ckpt) {
            if (__syncthreads_or(!r4_wait())) { failed = true; break; }
            const int jc = (c + 1) / p.ck_chunks - 1;
            float* dst = p.ckpt + ((size_t)blockIdx.x * p.n_ckpt + jc) * DIO * DIO + lane;
#pragma unroll
            for (int cc = 0; cc < 32; cc += 16) {
                float x[16];
                tmem_ld16(tq + TM_S + 32 * u + cc, x);  // warp-collective: every warp loads
#pragma unroll
                for (int jj = 0; jj < 16; jj++)
                    if (DIO == kD || (lane < DIO && 32 * u + cc + jj < DIO))
                        dst[(size_t)(32 * u + cc + jj) * DIO] = x[jj];
            }
            tc_fence_before();
        }
    }

    if (!failed && r4_pending && __syncthreads_or(!r4_wait())) failed = true;
    if (failed) flags |= KDA_DEV_TIMEOUT;
    // O rows of the last chunk.
    if (nchunks > 0 && !failed && !zero_exit) {
        store_o(nchunks - 1, min(kC, T - t_begin - (nchunks - 1) * kC));
        if (kind == 0) {
            fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0) {
                tma_store_4d(&map_o, sm + OFF_OST, 0, h, t_begin + (nchunks - 1) * kC, b);
                bulk_wait_all();
            }
        }
    }
    // Final state: hT (whole sequences), the segment's zero-start state or
    // its transition (segment pass), nothing (correction pass); in the
    // balanced schedule a head's state goes to its handoff slot.
    float* hTp = nullptr;
    {
        int bh2, seg2;
        task_seq(&bh2, &seg2);
        if (bal) hTp = to_slot ? p.bal_states + (size_t)bh * kD * kD
                       : p.hT  ? p.hT + (size_t)bh * DIO * DIO
                               : nullptr;
        else if (!SEG || p.pass == 0) hTp = p.hT ? p.hT + (size_t)bh2 * DIO * DIO : nullptr;
        else if (p.pass == 3) hTp = p.ws_m + (size_t)bh2 * kD * kD;
        else if (p.pass == 4) hTp = nullptr;
        else if (kind == 0) hTp = p.ws_s0 + ((size_t)bh2 * nseg + seg2) * kD * kD;
        else if (kind == 1) hTp = p.ws_m + ((size_t)bh2 * (nseg - 1) + seg2 - 1) * kD * kD;
    }
    if (hTp && !failed) {
        // the caller's hT at stride DIO; the handoff slots and the segment
        // workspace at kD (the segmented passes run only at DIO = kD)
        const int ld = to_slot ? kD : DIO;
        float* dst = hTp + lane;
#pragma unroll
        for (int cc = 0; cc < 32; cc += 16) {
            float x[16];
            tmem_ld16(tq + TM_S + 32 * u + cc, x);  // warp-collective: every warp loads
#pragma unroll
            for (int jj = 0; jj < 16; jj++)
                if (DIO == kD || (lane < ld && 32 * u + cc + jj < ld))
                    dst[(size_t)(32 * u + cc + jj) * ld] = x[jj];
        }
    }
    gc += nchunks;
    // The next task overwrites the state in TMEM and the O staging rows.
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (to_slot && tid == 0 && !failed) {
        __threadfence();
        st_release_gpu(p.bal_flags + bh, 1);
    }
    }  // tasks
    if (tid == kR2Thread) bulk_wait_all();
    report_flags(p.d_status, flags);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tbase, TM_COLS);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

// 4-D map over [B, T, H, d] (innermost first: d, H, T, B), boxes of
// box_inner x 1 x 64 x 1 with the 128-byte swizzle. Rows past T read as zero.
bool make_map(CUtensorMap* m, const void* ptr, CUtensorMapDataType dt, int esz, int B, int T,
              int H, int d, int box_inner,
              CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)d * esz, (cuuint64_t)H * d * esz,
                             (cuuint64_t)T * H * d * esz};
    cuuint32_t box[4] = {(cuuint32_t)box_inner, 1, (cuuint32_t)kC, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, dt, 4, const_cast<void*>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

namespace {

struct TcMaps {
    CUtensorMap q{}, k{}, v{}, g{}, o{};
};

bool make_maps(TcMaps* m, const ChunkFwdArgs& a) {
    if (a.T == 0) return true;
    // The caller's channel count (128, or 64 with the boxes still covering
    // 128 channels: zero-filled past the tensor on load, clipped on store).
    const int d = a.dk;
    return make_map(&m->q, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.B, a.T, a.H, d, 64) &&
           make_map(&m->k, a.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.B, a.T, a.H, d, 64) &&
           make_map(&m->v, a.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.B, a.T, a.H, d, 64) &&
           make_map(&m->g, a.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.B, a.T, a.H, d, 32) &&
           (!a.o || make_map(&m->o, a.o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.B, a.T, a.H, d, kD,
                             CU_TENSOR_MAP_SWIZZLE_NONE));
}

TcParams base_params(const ChunkFwdArgs& a) {
    TcParams p{a.beta, a.h0, static_cast<__nv_bfloat16*>(a.o), a.hT, a.T, a.H, a.d_status,
               a.ckpt, a.ckpt ? a.ckpt_every / kC : 1, a.ckpt ? a.T / a.ckpt_every : 0};
    p.pass = 0;
    p.nseg = 1;
    p.seg_chunks = 0;
    p.lead = 1;
    p.BH = a.B * a.H;
    p.ws_s0 = p.ws_m = nullptr;
    p.ws_sin = nullptr;
    p.bal_W = 0;
    p.bal_states = nullptr;
    p.bal_flags = nullptr;
    p.plan = nullptr;
    return p;
}

// dependent: launch as a programmatic dependent of the stream's previous
// kernel (its launch overlaps that kernel's end; the kernel waits for it).
template <bool SEG, int DIO = kD>
cudaError_t launch_tc(const TcMaps& m, const TcParams& p, long long grid, cudaStream_t stream,
                      bool dependent = false) {
    cudaError_t e = cudaFuncSetAttribute(kda_chunk_tc_kernel<SEG, DIO>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    if (!dependent) {
        kda_chunk_tc_kernel<SEG, DIO><<<(unsigned)grid, kThreads, SMEM_BYTES, stream>>>(
            m.q, m.k, m.v, m.g, m.o, p);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kda_chunk_tc_kernel<SEG, DIO>, m.q, m.k, m.v, m.g, m.o, p);
}

// Balanced schedule (see TcParams::bal_W): when B * H sequences do not fill
// whole waves of one CTA per SM, one cooperative launch of (at most) one CTA
// per SM gives every CTA the same number of chunk steps. Returns
// cudaErrorNotSupported when the plain schedule should run instead.
template <int DIO>
cudaError_t launch_balanced(const TcMaps& m, const ChunkFwdArgs& a) {
    if (!a.bal_ws || a.ckpt || a.T <= 0) return cudaErrorNotSupported;
    int dev = 0, nsm = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaFuncSetAttribute(kda_chunk_tc_kernel<false, DIO>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kda_chunk_tc_kernel<false, DIO>, kThreads,
                                                      SMEM_BYTES) != cudaSuccess ||
        nsm <= 0 || per_sm <= 0) {
        cudaGetLastError();
        return cudaErrorNotSupported;
    }
    const long long G = (long long)nsm * per_sm, BH = (long long)a.B * a.H;
    const long long nch = (a.T + kC - 1) / kC;
    if (BH <= G) return cudaErrorNotSupported;
    const long long W = (BH * nch + G - 1) / G;  // > nch: a range holds at most one head and one tail
    // Critical path in chunk steps: waves of whole sequences against W plus
    // about two chunk steps for each of the (at most two) state handoffs.
    const long long plain = ((BH + G - 1) / G) * nch;
    if ((W + 4) * 100 >= plain * 97) return cudaErrorNotSupported;
    TcParams p = base_params(a);
    p.bal_W = (int)W;
    p.bal_states = static_cast<float*>(a.bal_ws);
    p.bal_flags = reinterpret_cast<int*>(static_cast<char*>(a.bal_ws) +
                                         (size_t)BH * kD * kD * sizeof(float));
    cudaError_t e = cudaMemsetAsync(p.bal_flags, 0, (size_t)BH * sizeof(int), a.stream);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((BH * nch + W - 1) / W));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: a tail may wait on a head
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kda_chunk_tc_kernel<false, DIO>, m.q, m.k, m.v, m.g, m.o, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return cudaErrorNotSupported;
    }
    return cudaSuccess;
}

template <int DIO>
cudaError_t launch_whole(const ChunkFwdArgs& a) {
    TcMaps m;
    if (!make_maps(&m, a)) return cudaErrorInvalidValue;
    const cudaError_t e = launch_balanced<DIO>(m, a);
    if (e != cudaErrorNotSupported) return e;
    return launch_tc<false, DIO>(m, base_params(a), (long long)a.B * a.H, a.stream);
}

}  // namespace

cudaError_t launch_chunk_fwd_tc(const ChunkFwdArgs& a) {
    if (a.dv != a.dk) return launch_chunk_fwd_simt(a, KDA_BF16);
    if (a.dk == kD) return launch_whole<kD>(a);
    if (a.dk == 64) return launch_whole<64>(a);
    return launch_chunk_fwd_simt(a, KDA_BF16);
}

cudaError_t launch_chunk_fwd_tc_slice(const ChunkFwdArgs& a, int which, float* state) {
    TcMaps m;
    if (!make_maps(&m, a)) return cudaErrorInvalidValue;
    TcParams p = base_params(a);
    p.hT = nullptr;
    p.ckpt = nullptr;
    p.pass = which == 1 ? 3 : 4;
    if (which == 1) p.ws_m = state;
    else p.ws_sin = state;
    return launch_tc<true>(m, p, (long long)a.B * a.H, a.stream);
}

cudaError_t launch_chunk_fwd_tc_segmented(const ChunkFwdArgs& a, int nseg, int seg_chunks,
                                          int lead, float* ws) {
    if (nseg <= 1) return launch_chunk_fwd_tc(a);
    TcMaps m;
    if (!make_maps(&m, a)) return cudaErrorInvalidValue;
    const long long BH = (long long)a.B * a.H;
    const size_t DD = (size_t)kD * kD;
    float* s0 = ws;
    float* mt = s0 + (size_t)BH * nseg * DD;
    float* sin = mt + (size_t)BH * (nseg - 1) * DD;
    TcParams p = base_params(a);
    p.nseg = nseg;
    p.seg_chunks = seg_chunks;
    p.lead = lead;
    p.ws_s0 = s0;
    p.ws_m = mt;
    p.ws_sin = sin;
    p.hT = nullptr;  // the final state comes out of the scan
    p.pass = 1;
    cudaError_t e = launch_tc<true>(m, p, BH * (2 * nseg - 1), a.stream);
    if (e != cudaSuccess) return e;
    e = launch_segment_scan(s0, mt, sin, a.hT, (int)BH, nseg, a.stream);
    if (e != cudaSuccess) return e;
    p.pass = 2;
    return launch_tc<true>(m, p, BH * (nseg - 1), a.stream, true);
}

cudaError_t launch_chunk_fwd_tc_segmented_planned(const ChunkFwdArgs& a, int nseg_max,
                                                  float* ws, const int* plan) {
    TcMaps m;
    if (!make_maps(&m, a)) return cudaErrorInvalidValue;
    const long long BH = (long long)a.B * a.H;
    const size_t DD = (size_t)kD * kD;
    // Regions sized for nseg_max segments, indexed with the plan's count.
    float* s0 = ws;
    float* mt = s0 + (size_t)BH * nseg_max * DD;
    float* sin = mt + (size_t)BH * (nseg_max - 1) * DD;
    TcParams p = base_params(a);
    p.nseg = nseg_max;
    p.plan = plan;
    p.ws_s0 = s0;
    p.ws_m = mt;
    p.ws_sin = sin;
    p.hT = nullptr;  // the final state comes out of the scan
    p.pass = 1;
    cudaError_t e = launch_tc<true>(m, p, BH * (2 * nseg_max - 1), a.stream, true);
    if (e != cudaSuccess) return e;
    e = launch_segment_scan_planned(s0, mt, sin, a.hT, (int)BH, nseg_max, plan, a.stream);
    if (e != cudaSuccess) return e;
    p.pass = 2;
    return launch_tc<true>(m, p, BH * (nseg_max - 1), a.stream, true);
}

}  // namespace kda
