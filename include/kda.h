/*
 * kda.h — C ABI of the GB300 (sm_103a) Kimi Delta Attention (KDA) library.
 *
 * KDA is the linear-attention layer of the Kimi K3 architecture described on
 * the orkas.ai page "Kimi K3 architecture" (and its translations; the poyo.ai
 * page "Kimi K3 architecture" summarises it under "What is Kimi Delta
 * Attention?"). Per head it keeps a fixed-size state S (dk x dv, fp32) with a
 * per-channel decay and a token-dependent transition:
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t
 *
 * (section "Sequence: three quarters of the layers stopped reading
 * everything": a fixed-size state that decays; section "The bill arrives in
 * the serving stack": serial update, token-dependent transition of the
 * incoming state, in-place update while decoding). The log-decay is bounded,
 * g in [-5, 0] (section "A lower bound that deleted a GPU code path": at
 * least 0.67% of the state survives each step, so a 16-token tile's
 * cumulative log-decay stays above -80).
 *
 * Conventions shared by every entry point
 *   - Every data pointer is a DEVICE pointer owned by the caller. The library
 *     never allocates, frees or synchronises; work is enqueued on `stream`
 *     (a cudaStream_t passed as void*; NULL means the legacy default stream).
 *   - Tensors are contiguous and row-major; every pointer is 16-byte aligned
 *     except beta, which needs 4 bytes:
 *       q, k, g : [B, T, H, dk]      v, o : [B, T, H, dv]      beta : [B, T, H]
 *       h0, hT  : [B, H, dk, dv]     (decode: T = 1 and B = N, S = [N, H, dk, dv])
 *   - q, k, v, o have type `io` (bf16 or fp32); g, beta and states are fp32.
 *   - No scaling is applied to q: o = S^T q exactly. Callers that want
 *     1/sqrt(dk) pre-scale q.
 *   - Supported sizes: dk = dv in {64, 128}; any T >= 0 (ragged tails are
 *     handled; T = 0 writes hT = h0); B, H, N >= 0 (zero launches nothing)
 *     with B*H < 2^31, N*H < 2^30 and every tensor under 2^62 elements.
 *
 * Errors
 *   - Argument errors are reported synchronously by the return value and
 *     nothing is launched.
 *   - A failed launch returns KDA_ERR_CUDA; kda_last_error_string() then
 *     names the CUDA error (the library links its own CUDA runtime, so the
 *     caller's cudaGetLastError does not see it).
 *   - Data-dependent conditions are OR-ed, as the KDA_DEV_* bits below, into
 *     the device int `*d_status` when d_status is not NULL. The computation
 *     still runs to completion. The caller reads the word after its own
 *     synchronisation and clears it before reuse.
 */
#ifndef KDA_H_
#define KDA_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KDA_ABI_VERSION 2

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1, /* NULL pointer, bad size, misaligned pointer */
    KDA_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. dk != dv) */
    KDA_ERR_WORKSPACE = 3,   /* workspace pointer or size too small */
    KDA_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
    KDA_ERR_DECAY_RANGE = 5, /* (device) some g outside [-5, 0] */
    KDA_ERR_NONFINITE = 6,   /* (device) NaN or Inf in an input */
    KDA_ERR_TIMEOUT = 7      /* (device) a bounded on-chip wait gave up */
} kda_status_t;

typedef enum { KDA_BF16 = 0, KDA_F32 = 1 } kda_dtype_t;

/* Bits OR-ed into *d_status by the kernels. */
#define KDA_DEV_DECAY_RANGE 0x1 /* some g < -5 or g > 0 */
/* Some q, k, v, g or beta is NaN or Inf. g and beta are checked as they are
 * read; the decode kernels also check q, k and v as they are read. The
 * prefill kernels find a NaN or Inf in q, k or v through the outputs: any
 * of them makes some o non-finite through the recurrence, so they check
 * every o they compute (which also catches a non-finite h0 or an o that
 * overflows fp32). */
#define KDA_DEV_NONFINITE 0x2
#define KDA_DEV_TIMEOUT 0x4     /* an mbarrier wait exceeded its iteration cap */

/* Version of this header the library was built from (KDA_ABI_VERSION). */
int kda_abi_version(void);

/* Static string naming a status code; never NULL. */
const char* kda_status_string(kda_status_t s);

/* Why the last call on this host thread failed ("" if none did); never NULL. */
const char* kda_last_error_string(void);

/*
 * Bytes of device workspace that let kda_chunk_fwd balance the work over the
 * SMs: B*H*128*128*4 bytes of states plus B*H ints (rounded up to 256 bytes)
 * for io = KDA_BF16 (dk = dv = 64 or 128), T > 0 and B*H >= 2; 0 otherwise (the fp32
 * path keeps nothing off chip). With a buffer of at least this size the
 * tensor-core path may run one CTA per SM over the sequences laid end to end,
 * a sequence split between two CTAs handing its state over through the
 * buffer (it does so when B*H sequences would leave a partly filled last wave
 * of one CTA per sequence). A smaller buffer or NULL is accepted and runs one
 * CTA per sequence; both give bit-identical results. The buffer must be
 * 16-byte aligned, must not overlap any other argument and must not be used by
 * another call in flight; its contents need no initialisation.
 * Returns (size_t)-1 for arguments kda_chunk_fwd would reject.
 */
size_t kda_chunk_fwd_workspace_size(int B, int T, int H, int dk, int dv, kda_dtype_t io);

/*
 * Chunked forward (prefill) of KDA over B sequences of T tokens and H heads.
 *
 * Computes, for every (b, h), the recurrence above over t = 0..T-1 starting
 * from S_{-1} = h0[b, h] (zeros when h0 is NULL), writes o[b, t, h, :] = o_t
 * and, when hT is not NULL, hT[b, h] = S_{T-1}. Internally the sequence is
 * processed in chunks with 16-token decay tiles (the "divide by the
 * accumulated decay" blockwise evaluation of section "A lower bound that
 * deleted a GPU code path"); the result equals the token-by-token recurrence
 * up to rounding.
 *
 *   q, k   : [B, T, H, dk] of type io          (in)
 *   v      : [B, T, H, dv] of type io          (in)
 *   g      : [B, T, H, dk] fp32 log-decay      (in; must lie in [-5, 0])
 *   beta   : [B, T, H]     fp32                (in)
 *   h0     : [B, H, dk, dv] fp32 or NULL       (in)
 *   o      : [B, T, H, dv] of type io          (out; must not alias inputs)
 *   hT     : [B, H, dk, dv] fp32 or NULL       (out; may alias h0)
 *   workspace, ws_bytes : see kda_chunk_fwd_workspace_size
 *   d_status : device int or NULL              (in/out, OR-ed KDA_DEV_* bits)
 *   stream : cudaStream_t
 *
 * io = KDA_BF16 runs the tensor-core (tcgen05/TMEM) path with fp32 state; at
 * dk = dv = 64 it runs as dk = dv = 128 with channels 64..127 zero (the tensor
 * maps fill them with zeros on load and clip them on store, so the bytes moved
 * are those of d = 64 and the zero channels add only exact zeros to every sum;
 * the arithmetic is that of d = 128). io = KDA_F32 runs an fp32 CUDA-core path, untuned,
 * meant for accuracy rather than speed. With a
 * full-size workspace the tensor-core path enqueues a memset of the handoff
 * flags before its (cooperative) launch.
 */
kda_status_t kda_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                           const float* beta, const float* h0, void* o, float* hT, int B,
                           int T, int H, int dk, int dv, kda_dtype_t io, void* workspace,
                           size_t ws_bytes, int* d_status, void* stream);

/*
 * kda_chunk_fwd that also saves the state at sparse boundaries: the state
 * after token (j + 1) * ckpt_every - 1 goes to ckpt[b, h, j] for
 * j = 0 .. T / ckpt_every - 1 (section "The bill arrives in the serving
 * stack", second bullet: prefix reuse hashes every 512 tokens but keeps a
 * recurrent-state restore point only at a sparse subset of those boundaries).
 *
 *   ckpt       : [B, H, T / ckpt_every, dk, dv] fp32 (out; must not overlap
 *                any other tensor); the last entry equals hT when ckpt_every
 *                divides T
 *   ckpt_every : positive multiple of 64 (the chunk length), e.g. 512 or 2048
 *
 * Other arguments as for kda_chunk_fwd (no workspace is needed). Each
 * checkpoint adds dk * dv * 4 bytes of writes per (b, h).
 */
kda_status_t kda_chunk_fwd_ckpt(const void* q, const void* k, const void* v, const float* g,
                                const float* beta, const float* h0, void* o, float* hT,
                                float* ckpt, int ckpt_every, int B, int T, int H, int dk, int dv,
                                kda_dtype_t io, int* d_status, void* stream);

/*
 * kda_chunk_fwd with every sequence split in time into segments that run in
 * parallel, for few long sequences (B * H well below the SM count). Section
 * "The bill arrives in the serving stack", first bullet: the incoming state
 * of a segment is not a sum of per-segment states, but each segment has two
 * composable summaries, its cumulative transition M (the product of its
 * per-token transitions) and its final state S0 from a zero start, and a
 * prefix scan over them rebuilds every segment's incoming state. Here: a
 * segment pass (every segment from a zero start, the first from h0, writing
 * o; segments after the first also from the identity with v = 0, giving M),
 * the scan X_{s+1} = S0_s + M_s X_s in fp32 (its last value is hT), and a
 * correction pass (segments after the first again, from X_s with v = 0,
 * adding their outputs to o). o and hT equal kda_chunk_fwd's up to rounding
 * (o of later segments is the sum of two bf16-rounded parts).
 *
 *   nseg      : segments per sequence, 1 .. ceil(T / 64); 1 runs
 *               kda_chunk_fwd. 0: planned on the device from the data:
 *               kda_chunk_fwd_decay_probe's statistic of g is reduced by a
 *               planning kernel to the split kda_chunk_fwd_segments_hint_decay
 *               would choose (up to min(32, ceil(T / 64)) segments), and the
 *               passes read it from device memory; five launches, no host
 *               synchronisation (so it can be captured into a CUDA graph); B
 *               must be <= 65535 and lead <= 0; with fewer than two chunks
 *               it runs kda_chunk_fwd. As many segments result as an even split into
 *               ceil(ceil(T / 64) / nseg)-chunk segments leaves non-empty
 *               (at most nseg); the first, which needs no transition and no
 *               correction, may span several segment lengths so that its long
 *               runs overlap the other segments' passes on the remaining SMs
 *               (kda_chunk_fwd_segment_plan gives the split for the device)
 *   lead      : the first segment's length in segment lengths, 1 ..
 *               ceil(T / 64), or <= 0 for the library's choice (the length
 *               kda_chunk_fwd_segment_plan reports for lead <= 0); a lead
 *               that leaves fewer non-empty segments runs fewer.
 *               kda_chunk_fwd_segments_hint_decay suggests nseg and lead
 *               together. The results do not depend on the split beyond
 *               rounding.
 *   workspace : device buffer of kda_chunk_fwd_segmented_workspace_size bytes,
 *               16-byte aligned, not overlapping any other tensor; contents
 *               are scratch
 *
 * Other arguments as for kda_chunk_fwd. Needs io = KDA_BF16 and
 * dk = dv = 128 when it splits (KDA_ERR_UNSUPPORTED otherwise); a missing or
 * short workspace returns KDA_ERR_WORKSPACE. The split part costs about three
 * times the arithmetic of one pass; kda_chunk_fwd_segments_hint says when it
 * pays.
 */
kda_status_t kda_chunk_fwd_segmented(const void* q, const void* k, const void* v,
                                     const float* g, const float* beta, const float* h0, void* o,
                                     float* hT, int B, int T, int H, int dk, int dv,
                                     kda_dtype_t io, int nseg, int lead, void* workspace,
                                     size_t ws_bytes, int* d_status, void* stream);

/*
 * Bytes of workspace kda_chunk_fwd_segmented needs: (3 nseg' - 2) * dk * dv * 4
 * per (b, h), nseg' the number of segments that results, 0 when that is 1.
 * For nseg = 0 (planned on the device): the same for nseg' = min(32,
 * ceil(T / 64)), plus 16 * B * H floats of probe (rounded up to 16 bytes) and
 * 16 bytes of plan (0 with fewer than two chunks). Returns (size_t)-1 for
 * arguments kda_chunk_fwd_segmented would reject.
 */
size_t kda_chunk_fwd_segmented_workspace_size(int B, int T, int H, int dk, int dv,
                                              kda_dtype_t io, int nseg);

/*
 * kda_chunk_fwd_segmented for callers that cannot allocate device memory: the
 * call takes no workspace and allocates nothing. Such callers include
 * serving runtimes that reserve all device memory up front and hand the
 * library none of it, and memory-pool or allocator plugins that must not call
 * back into the allocator that is running them. The paper has no
 * counterpart: this is a deployment variant of kda_chunk_fwd_segmented.
 *
 * The scratch is a 48 MB array in the library's own device image; every GPU
 * that loads the library holds one copy until the process exits. Its device
 * address is looked up once per device, by the first call of this function on
 * that device (with the device current); make that first call before any
 * stream capture. Limits and sharing:
 *   - kda_chunk_fwd_segmented_workspace_size(B, T, H, dk, dv, io, nseg) must
 *     be at most 48 MB, i.e. B * H * (3 nseg' - 2) <= 768 with nseg' the
 *     number of segments that results (e.g. nseg <= 8 at B = 1, H = 32;
 *     nseg <= 6 at B * H = 48). The count kda_chunk_fwd_segments_hint
 *     returns can exceed this (it does at B = 1, T = 2^20, H = 32): pass a
 *     smaller nseg here. A larger problem returns KDA_ERR_WORKSPACE before
 *     any launch.
 *   - Every call on a device shares the array: calls whose work overlaps on
 *     the GPU (different streams, or host threads) race and give wrong
 *     results; serialise them on one stream. The array keeps the last call's
 *     contents; nothing in it needs to start at zero (every value is written
 *     before it is read).
 * Argument errors are checked first, as for kda_chunk_fwd_segmented; other
 * arguments, results and errors are those of kda_chunk_fwd_segmented.
 */
kda_status_t kda_chunk_fwd_segmented_noalloc(const void* q, const void* k, const void* v,
                                             const float* g, const float* beta, const float* h0,
                                             void* o, float* hT, int B, int T, int H, int dk,
                                             int dv, kda_dtype_t io, int nseg, int lead,
                                             int* d_status, void* stream);

/*
 * Segment count that minimises the number of chunk steps on the critical
 * path on the current device (one CTA per SM, whole sequences against the
 * segment and correction passes), or 1 when splitting does not save at
 * least a fifth; 1 also when no CUDA device is visible or the configuration
 * has no segmented path. -1 for arguments kda_chunk_fwd would reject.
 */
int kda_chunk_fwd_segments_hint(int B, int T, int H, int dk, int dv, kda_dtype_t io);

/*
 * Sampled decay statistic for planning a split in time. A run with v = 0 (a
 * segment's transition from the identity, a correction from its incoming
 * state) multiplies its state token by token by (I - b k k^T) Diag(e^g); for
 * unit keys and 0 <= b <= 2 the first factor is a contraction, so over a
 * 64-token chunk the state's entries shrink at least by
 * e^{sum_t max_c g[t, c]}, and once they pass fp32's smallest subnormal the
 * state is exactly zero and the segmented prefill stops that run. This call
 * writes d_probe[(b * nsample + s) * H + h] = sum_t max_c g[b, t, h, c] over
 * the tokens t of chunk floor(s * nch / nsample) of batch row b
 * (nch = ceil(T / 64); a short last chunk sums its tokens only).
 *   g        : [B, T, H, dk] fp32 device, 16-byte aligned (the prefill's g)
 *   nsample  : chunks sampled per batch row, 1 .. 4096
 *   d_probe  : device, B * nsample * H floats, 4-byte aligned, not
 *              overlapping g
 * One launch of B * nsample * ceil(H / 8) CTAs on `stream`, four warps per
 * (sample, row, head) reading 16 of that head's 64 rows of dk floats each; nothing
 * written when B, H or T is 0. dk must be 64 or 128 (KDA_ERR_UNSUPPORTED),
 * B <= 65535, H <= 524280. The statistic guides the plan only: the results
 * of the segmented call never depend on it.
 */
kda_status_t kda_chunk_fwd_decay_probe(const float* g, int B, int T, int H, int dk, int nsample,
                                       float* d_probe, void* stream);

/*
 * kda_chunk_fwd_segments_hint with a decay statistic: probe (host memory,
 * nprobe floats, e.g. a copy of kda_chunk_fwd_decay_probe's output) gives the
 * decay per chunk the sequences can be counted on (its largest entry, cd).
 * With cd < 0 the planner counts each transition and correction run as
 * stopping after about 2 + ceil(103.28 / -cd) chunks instead of running its
 * whole segment, which favours more, shorter segments and a shorter first
 * one; with no entries, an entry >= 0 or a non-finite entry it plans as
 * kda_chunk_fwd_segments_hint. Returns the segment count (1 = do not split)
 * and writes the matching lead to *lead (if not NULL; 1 when it returns 1);
 * pass both to kda_chunk_fwd_segmented. A sample that misses slowly decaying
 * stretches makes those runs longer than planned: slower, never different
 * results. -1 for arguments kda_chunk_fwd would reject, nprobe < 0 or a NULL
 * probe with nprobe > 0.
 */
int kda_chunk_fwd_segments_hint_decay(int B, int T, int H, int dk, int dv, kda_dtype_t io,
                                      const float* probe, int nprobe, int* lead);

/*
 * The split kda_chunk_fwd_segmented uses for nseg and lead_in (its lead
 * argument; <= 0: the library's choice) on the current device: returns the
 * number of segments that results (1 = no split), or -1 for arguments
 * kda_chunk_fwd_segmented would reject and for nseg = 0 (that split is
 * chosen on the device from the data). *seg_chunks (if not NULL)
 * receives the length of every segment after the first in 64-token chunks
 * (the last may be shorter; ceil(T / 64) when there is no split) and *lead
 * (if not NULL) the first segment's length in those units. The first segment
 * length is lead_in when positive, else the one of 1 .. 16 that minimises
 * the chunk steps on the critical path when the segment pass starts the
 * first segments' long runs on B * H SMs and the other runs on the rest,
 * counting every run as its whole segment; 1 when no CUDA device is visible.
 */
int kda_chunk_fwd_segment_plan(int B, int T, int H, int dk, int dv, kda_dtype_t io, int nseg,
                               int lead_in, int* seg_chunks, int* lead);

/*
 * Building blocks for one long sequence split in time across devices (or
 * processes): section "The bill arrives in the serving stack", first bullet,
 * of the orkas.ai page "Kimi K3 architecture". The incoming state of a later
 * time slice is not a sum of per-slice states, but every slice has two
 * composable summaries: its cumulative transition M (the product of its
 * per-token transitions (I - b k k^T) Diag(e^g)) and its final state S0 from a
 * zero start; a prefix scan over them rebuilds every slice's incoming state
 * after one fixed-size exchange of the summaries. With the time slices
 * numbered 0 .. n-1, each on its own device:
 *   1. kda_chunk_fwd on the slice (slice 0 from h0, the others from zero)
 *      writes o and S0; kda_chunk_fwd_slice_transition writes M (slices > 0);
 *   2. the (S0, M) pairs of all slices are gathered on every device;
 *   3. kda_state_scan turns them into the incoming state of every slice and
 *      the sequence's final state;
 *   4. kda_chunk_fwd_slice_correct adds, on slices > 0, the outputs that the
 *      incoming state contributes.
 * The package's seqsplit.py runs these steps over a torch.distributed group.
 * All three need io = KDA_BF16 and dk = dv = 128 (KDA_ERR_UNSUPPORTED
 * otherwise); tensors as for kda_chunk_fwd, [B, T, H, dk] for the slice.
 */

/*
 * M[b, h] = the product of the slice's per-token transitions (the recurrence
 * run from the identity with v = 0): [B, H, dk, dk] fp32, out, must not
 * overlap the inputs; the identity when T = 0. q and k are of type io; g and
 * beta fp32. d_status and stream as for kda_chunk_fwd.
 */
kda_status_t kda_chunk_fwd_slice_transition(const void* q, const void* k, const float* g,
                                            const float* beta, float* M, int B, int T, int H,
                                            int dk, kda_dtype_t io, int* d_status, void* stream);

/*
 * o += the outputs of the recurrence over the slice run from S_in with v = 0,
 * i.e. what the slice's incoming state adds to the outputs of its zero-start
 * run. S_in: [B, H, dk, dv] fp32 (in); o: [B, T, H, dv] of type io (in/out,
 * must not overlap the inputs or S_in). Other arguments as above.
 */
kda_status_t kda_chunk_fwd_slice_correct(const void* q, const void* k, const float* g,
                                         const float* beta, const float* S_in, void* o, int B,
                                         int T, int H, int dk, int dv, kda_dtype_t io,
                                         int* d_status, void* stream);

/*
 * Prefix scan over the summaries of nslice consecutive time slices, all fp32:
 *   s0   : [nslice, B, H, dk, dv]      final states from a zero start (slice
 *                                      0's from the sequence's initial state)
 *   m    : [nslice - 1, B, H, dk, dk]  transitions of slices 1 .. nslice - 1
 *   x_in : [nslice - 1, B, H, dk, dv]  out: incoming state of slices 1 ..
 *   hT   : [B, H, dk, dv] or NULL      out: the sequence's final state
 * X_1 = s0[0], X_{s+1} = s0[s] + m[s - 1] X_s. m and x_in may be NULL when
 * nslice = 1. Outputs must not overlap the inputs or each other.
 */
kda_status_t kda_state_scan(const float* s0, const float* m, float* x_in, float* hT, int nslice,
                            int B, int H, int dk, int dv, void* stream);

/*
 * Self-test of failure detection. Every wait of the kernels above on an
 * mbarrier (TMA arrival, MMA completion) is a bounded loop: when it gives up
 * (~2^31 SM clocks) the kernel ORs KDA_DEV_TIMEOUT into *d_status, stops, frees
 * its tensor memory and returns, so a stuck pipeline surfaces as a status
 * instead of a hung GPU. This launches one CTA that runs the same bounded
 * wait on an mbarrier that nothing ever completes, giving up after `clocks`
 * SM clocks (1 .. 2^31), and ORs KDA_DEV_TIMEOUT into *d_status (device int,
 * required). The context stays usable afterwards.
 */
kda_status_t kda_selftest_wait_timeout(long long clocks, int* d_status, void* stream);

/*
 * One decode step for N sequences (one token each), state updated in place
 * (section "The bill arrives in the serving stack", third bullet: the state
 * is overwritten where it lives).
 *
 *   q, k : [N, H, dk] of type io;  v : [N, H, dv] of type io
 *   g    : [N, H, dk] fp32;        beta : [N, H] fp32
 *   S    : [N, H, dk, dv] fp32, read as S_{t-1} and overwritten with S_t
 *   o    : [N, H, dv] of type io,  o = S_t^T q
 *   d_status, stream : as for kda_chunk_fwd
 *
 * HBM-bandwidth bound: each call reads and writes S once.
 */
kda_status_t kda_decode_step(const void* q, const void* k, const void* v, const float* g,
                             const float* beta, float* S, void* o, int N, int H, int dk,
                             int dv, kda_dtype_t io, int* d_status, void* stream);

/*
 * Multi-token decode for speculative decoding: K cached tokens per sequence
 * applied to the state in one pass (section "The bill arrives in the serving
 * stack", third bullet: the state is overwritten in place, so a rejected draft
 * cannot be rolled back; the small projected inputs of the draft are cached
 * and the state is rebuilt on chip instead).
 *
 *   q, k, g : [N, K, H, dk] (q, k of type io; g fp32)
 *   v       : [N, K, H, dv] of type io;  beta : [N, K, H] fp32
 *   S       : [N, H, dk, dv] fp32, the state before token 0
 *   o       : [N, K, H, dv] of type io, o[n, t] = S_t^T q_t (tokens t < ntok[n])
 *   ntok    : device int[N] or NULL; sequence n takes its first
 *             min(max(ntok[n], 0), K) tokens (NULL: all K)
 *   commit  : 0 = verify: S is only read, o is written (o must not be NULL);
 *             1 = commit: S is overwritten with the state after ntok[n]
 *                 tokens; o is written when not NULL
 *
 * Typical use: verify the K draft tokens (commit = 0), accept m_n of them,
 * then commit with ntok = m (o = NULL). Each call reads the state once and
 * writes it at most once. Errors and d_status as for kda_decode_step.
 */
kda_status_t kda_decode_multi(const void* q, const void* k, const void* v, const float* g,
                              const float* beta, float* S, void* o, const int* ntok, int N, int K,
                              int H, int dk, int dv, kda_dtype_t io, int commit, int* d_status,
                              void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H_ */
