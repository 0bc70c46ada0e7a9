/*
 * libfa — exact attention on one GB300 GPU (sm_103a), C ABI.
 *
 *   O = softmax(scale * Q K^T) V
 *
 * computed FlashAttention-2 style: every CTA owns a block of query rows and
 * walks the keys in blocks, carrying a running row maximum m, denominator l and
 * unnormalised accumulator, so the score matrix never reaches device memory.
 *
 * Conventions shared by every call
 * --------------------------------
 * - All tensor pointers are DEVICE pointers owned by the caller, dense and
 *   contiguous, 16-byte aligned. The library allocates no device memory.
 * - Layout: Q, O, dO, dQ are [B, H, M, D]; K, V, dK, dV are [B, H, N, D]
 *   (row-major, D fastest). LSE and delta are [B, H, M] float32.
 * - dtype selects the storage type of Q/K/V/O/dO/dQ/dK/dV: FA_F16, FA_BF16 or
 *   FA_F32. Softmax state and accumulation are float32 in every case; the f32
 *   path contracts with three TF32 products (hi*hi + hi*lo + lo*hi).
 * - D must be 64 or 128 (FA_ERR_UNSUPPORTED otherwise).
 * - stream is a cudaStream_t (NULL = the legacy default stream). Calls are
 *   asynchronous: the return value covers argument checks and the launch only.
 *   Faults detected on the device (a bounded wait that ran out) are reported by
 *   fa_last_status() after the caller synchronises.
 * - Errors: FA_ERR_INVALID for bad arguments (null pointer, misaligned pointer,
 *   non-positive sizes, index overflow); nothing is launched in that case.
 *   fa_last_error_message() returns a one-line reason for the calling thread.
 * - B*H == 0 or M == 0 is an empty problem: FA_OK, nothing launched.
 */
#ifndef FA_H
#define FA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa_status {
  FA_OK = 0,
  FA_ERR_INVALID = 1,     /* bad argument, nothing launched */
  FA_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. D not in {64,128}) */
  FA_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed */
  FA_ERR_TIMEOUT = 4      /* a kernel gave up a bounded wait (see fa_last_status) */
} fa_status;

typedef enum fa_dtype { FA_F32 = 0, FA_F16 = 1, FA_BF16 = 2 } fa_dtype;

/*
 * Forward pass (prefill).
 *
 * Follows "Flash attention, f32" (Phobos examples: the online-softmax loop
 * over key blocks, "After the loop" normalisation) and "06: Fused attention"
 * (attn_fwd: causal rule, stored log-sum-exp L = m + log l).
 *
 *   Q [B,H,M,D], K [B,H,N,D], V [B,H,N,D]  inputs, dtype
 *   O [B,H,M,D]                            output, dtype (round to nearest even)
 *   LSE [B,H,M] float32                    output, natural log of the row sum of
 *                                          exp(scale*q.k); may be NULL
 *   scale                                  multiplies Q K^T before the softmax;
 *                                          any finite value (scale < 0 negates
 *                                          the score product in the tensor core)
 *   causal                                 nonzero: key j is visible to query i
 *                                          iff j <= i (top-left aligned)
 * M, N >= 1 (N == 0 is FA_ERR_INVALID). Any M, N: ragged tails are masked.
 */
fa_status fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int M, int N,
                 int D, float scale, int causal, fa_dtype dtype, void* stream);

/*
 * Bytes of device workspace fa_fwd_ws can use for this problem on the current
 * device. fp16/bf16 with D = 64 (causal or not): one partial-result slot (a
 * 256x64 f32 block and three 256-float statistics) plus eight 32-bit flags per
 * SM. f32 with D = 64 when its 128-row query tiles fill fewer than half the SMs:
 * one 128x64 f32 block plus two 128-float statistics per (tile, part), where the
 * key blocks of a tile are shared by `parts` SMs, then four 64-bit counters per
 * tile. Otherwise, or on bad sizes, 0.
 */
size_t fa_fwd_workspace_bytes(int B, int H, int M, int N, int D, int causal, fa_dtype dtype);

/*
 * fa_fwd with a caller-owned workspace; same arguments, same results.
 *
 * The pages' forward gives each CTA whole blocks of query rows. When the number
 * of 256-row query pairs does not fill the last wave of SMs, this call instead
 * gives every SM an equal contiguous share of (query pair, key block) work; a
 * pair whose key blocks are shared by two or more SMs is merged at the end by the
 * SM holding its first blocks, with the same (m, l) rescaling the online softmax
 * uses between key blocks. That SM waits (bounded, fa_set_wait_budget_ns) for the
 * flags of the SMs holding the rest, which process those pieces first; the
 * launch has one CTA per SM and relies on all of them becoming resident within
 * the wait budget, which holds unless kernels on other streams or processes
 * keep SMs busy for longer than that (then FA_ERR_TIMEOUT;
 * fa_set_schedule(FA_SCHED_FWD_SPLIT, 0) runs whole pairs, with no waits).
 * Every forward launch is a programmatic dependent of the kernel before it on
 * the stream: its set-up overlaps that kernel's tail.
 *
 *   workspace        device pointer, 16-byte aligned, at least
 *                    fa_fwd_workspace_bytes(...) bytes, or NULL (then this is
 *                    fa_fwd). Zero-filled by the caller before its first use;
 *                    afterwards the library leaves it in a reusable state
 *                    (flags carry a per-launch epoch from a sequence that
 *                    starts at a clock-drawn value, and consumed flags are
 *                    reset to zero). If other data were written over it,
 *                    zero-fill it again before the next call.
 *                    Owned by the caller; two calls must not use the same
 *                    workspace at the same time.
 *   workspace_bytes  its size; smaller than needed is FA_ERR_INVALID.
 *
 * The split is used when an estimate of its time in key blocks per SM (its
 * share, plus 3.5 for piece boundaries and the merge, plus 1.2 for each further
 * partial the holder of a pair's first blocks merges) is below 0.97 of whole
 * pairs' (non-causal: rounds x key blocks a pair; causal: the heaviest pair,
 * and only with fewer pairs than SMs, since from a round of pairs up causal
 * pairs dealt whole in a serpentine order measured faster);
 * fa_set_schedule(FA_SCHED_FWD_SPLIT, 0 or 1) turns it off or on regardless.
 * For f32 with few query tiles, several CTAs share each tile's keys: each writes
 * an unnormalised partial and counts itself in on the tile, and the one that
 * counts in last merges the partials the same way and writes O and LSE.
 */
fa_status fa_fwd_ws(const void* Q, const void* K, const void* V, void* O, float* LSE, void* workspace,
                    size_t workspace_bytes, int B, int H, int M, int N, int D, float scale, int causal, fa_dtype dtype,
                    void* stream);

/*
 * The forward on HOST buffers: copies in, computes and copies out, overlapped.
 *
 * For callers whose Q, K, V live in host memory and who want O (and LSE) back
 * there. The (batch, head) heads are cut into three chunks of about 4/7, 2/7
 * and 1/7 of them (equal chunks below seven heads; fa_set_schedule with
 * FA_SCHED_HOST_CHUNKS fixes a count of equal chunks instead, 1..8); the
 * library's own copy and compute streams for the device move chunk c in while
 * chunk c-1 is computed (same kernels and results as fa_fwd_ws) and earlier
 * chunks' outputs travel back. The call is asynchronous and ordered on `stream`: work queued
 * on `stream` before it happens first, and `stream` waits for the last copy
 * out before anything queued after it. Not for stream capture (the internal
 * streams and events are not part of a capture).
 *
 *   hQ [B,H,M,D], hK, hV [B,H,N,D]   host inputs, dtype; page-locked
 *                                     (cudaHostAlloc / cudaHostRegister) for
 *                                     the copies to overlap, else they stage
 *   hO [B,H,M,D]                      host output, dtype
 *   hLSE [B,H,M]                      host output, float32, or NULL
 *   dev_ws, dev_ws_bytes              device workspace of at least
 *                                     fa_fwd_host_workspace_bytes(...) bytes,
 *                                     16-byte aligned, zero-filled before its
 *                                     first use; it holds the device copies of
 *                                     Q, K, V, O, LSE and the forward's own
 *                                     workspace, whose place depends on the
 *                                     problem's shape, so zero-fill it again
 *                                     when the shape or dtype changes; two
 *                                     calls must not share it at the same time
 *   the rest                          as for fa_fwd
 * Errors as fa_fwd, plus FA_ERR_INVALID for a NULL host buffer or a small
 * workspace; arguments are checked before anything is queued.
 */
fa_status fa_fwd_host(const void* hQ, const void* hK, const void* hV, void* hO, float* hLSE, void* dev_ws,
                      size_t dev_ws_bytes, int B, int H, int M, int N, int D, float scale, int causal,
                      fa_dtype dtype, void* stream);

/* Bytes of device workspace fa_fwd_host needs (0 on bad sizes or dtype). */
size_t fa_fwd_host_workspace_bytes(int B, int H, int M, int N, int D, int causal, fa_dtype dtype);

/*
 * Backward pass: gradients of sum(dO o O).
 *
 * Follows "06: Fused attention" (attn_bwd_delta, attn_bwd_dkdv, attn_bwd_dq)
 * and the identity D_i = rowsum(dO o O), dS = P o (dP - D) from the "Flash
 * Attention" notes ("IO complexity"). Three launches on `stream`: delta, then
 * dK/dV (one CTA per key block walking the query blocks), then dQ (one CTA per
 * query block walking the key blocks). With D = 64, no causal mask and fewer
 * key tiles (B*H*ceil(N/128)) than SMs, the dK/dV and dQ launches run on CTA
 * pairs ("Flash Attention" notes, "FlashAttention 4": a 256-row tile split
 * across two CTAs with tcgen05 cta_group::2): each cluster of two CTAs owns 256
 * keys (dK/dV) or 256 queries (dQ), and one MMA covers both CTAs' rows with each
 * CTA holding half of the other operand (fa_set_schedule, FA_SCHED_BWD_PAIR).
 * dK and dV are bit-identical either way.
 *
 *   Q, K, V, O, dO   inputs (O from fa_fwd with the same arguments)
 *   LSE              input, [B,H,M] float32 written by fa_fwd
 *   dQ [B,H,M,D], dK [B,H,N,D], dV [B,H,N,D]   outputs, dtype
 *   delta_ws         caller-owned scratch of fa_bwd_workspace_bytes(B,H,M)
 *                    bytes; holds rowsum(dO o O) (float32 [B,H,M]) on return
 * dtype must be FA_F16 or FA_BF16 (FA_ERR_UNSUPPORTED for FA_F32: the page
 * that defines the f32 method, "Flash attention, f32", gives a forward only);
 * scale as for fa_fwd (any finite value; dK and dQ carry its sign).
 */
fa_status fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
                 void* dQ, void* dK, void* dV, float* delta_ws, int B, int H, int M, int N, int D, float scale,
                 int causal, fa_dtype dtype, void* stream);

/* Bytes of scratch fa_bwd needs: B*H*M float32. */
size_t fa_bwd_workspace_bytes(int B, int H, int M);

/*
 * fa_bwd with a caller-owned workspace that also holds an f32 dQ accumulator;
 * same arguments as fa_bwd (delta_ws replaced by workspace), same results.
 *
 * The pages' backward recomputes S and dP in a separate dQ kernel. With D = 64
 * this call instead forms dQ in the dK/dV pass: dS, already in shared memory
 * for dK += dS^T Q, also gives dQ_i = dS K, whose 128x64 block is added into an
 * f32 accumulator in global memory (a bulk reduce-add in L2); a last kernel
 * writes dQ = scale * accumulator in the I/O dtype. Five matrix products per
 * (query block, key block) instead of seven. For D = 128 it runs the three
 * kernels of fa_bwd.
 *
 *   workspace        device pointer, 16-byte aligned, at least
 *                    fa_bwd_ws_workspace_bytes(B,H,M,D) bytes: delta
 *                    (B*H*M float32, rowsum(dO o O) on return), then for
 *                    D = 64 the accumulator (B*H*M*64 float32, 256-byte
 *                    aligned), then per SM of the current device two slots
 *                    of partial dK/dV (2*64*128 float32 each) and, after all
 *                    slots, 8 counters (uint32) per SM. The call writes
 *                    every part it reads (no zero-fill needed); caller-owned,
 *                    one call at a time.
 *   workspace_bytes  its size; smaller than needed is FA_ERR_INVALID.
 * Non-causal calls with D = 64 may run a split schedule: every SM takes a
 * contiguous share of the (key tile, query block) pairs. The SMs holding the
 * later blocks of a cut key tile take those pieces first and write their
 * partial dK/dV; the SM holding its first blocks takes its piece last, waits
 * (bounded, fa_set_wait_budget_ns) until they have counted in, adds them and
 * writes the tile. The split is used when an estimate of its time in (key tile,
 * query block) steps per SM (its share, plus 5 for piece boundaries and the
 * merge, plus 0.8 per further partial a tile's first-block holder adds) is below
 * 0.97 of whole tiles' (rounds x ceil(M/128));
 * fa_set_schedule(FA_SCHED_BWD_SPLIT, 0 or 1) turns it off or on regardless.
 * The summation order of dQ's key blocks follows the SMs' timing, so dQ can
 * differ between runs in the last bits of the f32 accumulator, and so can dK
 * and dV of a key tile the split schedule cuts (otherwise they do not).
 */
fa_status fa_bwd_ws(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
                    void* dQ, void* dK, void* dV, void* workspace, size_t workspace_bytes, int B, int H, int M,
                    int N, int D, float scale, int causal, fa_dtype dtype, void* stream);

/* Bytes of workspace fa_bwd_ws needs (0 on bad sizes). */
size_t fa_bwd_ws_workspace_bytes(int B, int H, int M, int D);

/*
 * FP8 forward: the forward with both products on E4M3 operands.
 *
 * Follows "Flash Attention" (notes), section "FlashAttention 3", the FP8 bullets:
 * incoherent processing (Q and K multiplied on the right by M = diag(signs) H / 8,
 * H the 64 x 64 Hadamard matrix, so that (Q M)(K M)^T = Q K^T while outliers
 * spread over all 64 columns) and block quantisation (one scale per 128-row
 * block of Q M and of K M, scale = block max / 448). V has one scale per
 * (batch, head), because its key blocks are summed in one accumulator; the
 * softmax weights are rounded to E4M3 for P V; O is divided by the sum of the
 * rounded weights, LSE (natural log, f32) uses the exact sum. Two launches of
 * quantisation kernels into the workspace, then the attention kernel.
 *
 *   Q, K, V, O, LSE, B, H, M, N, scale, causal   as for fa_fwd
 *   D                  64 (other values: FA_ERR_UNSUPPORTED)
 *   dtype              FA_F16 or FA_BF16 (storage of Q, K, V, O)
 *   signs              device pointer, 16-byte aligned, to D signed bytes, each
 *                      +1 or -1 (a negative byte counts as -1), drawn by the
 *                      caller
 *   workspace          device pointer, 16-byte aligned, at least
 *                      fa_fwd_fp8_workspace_bytes(B,H,M,N,D) bytes: the E4M3
 *                      copies of Q M [B*H][M][64] and K M [B*H][N][64], V
 *                      transposed [B*H][64][N rounded up to 16], then the f32
 *                      scales; caller-owned, written before it is read (no
 *                      zero-fill needed), one call at a time
 * The results are approximations: RMSE of O about 2e-3 to 8e-3 against exact
 * attention on unit-variance inputs at scale 1/8.
 */
fa_status fa_fwd_fp8(const void* Q, const void* K, const void* V, void* O, float* LSE, const signed char* signs,
                     void* workspace, size_t workspace_bytes, int B, int H, int M, int N, int D, float scale,
                     int causal, fa_dtype dtype, void* stream);

/* Bytes of workspace fa_fwd_fp8 needs (0 on bad sizes or D != 64). */
size_t fa_fwd_fp8_workspace_bytes(int B, int H, int M, int N, int D);

/*
 * Decode (flash decoding): one query row per (batch, head) against a KV cache
 * (fa_decode_ex below takes up to four rows and returns the LSE too).
 *
 * Follows "Flash decoding" (linear algebra for programmers, part 4),
 * "Overview of the algorithm": the keys are cut into n_splits chunks of
 * ceil(N / n_splits) keys; each chunk s writes an UNNORMALISED partial
 *   m_s = max_j x_j,  l_s = sum_j e^{x_j - m_s},  O_s = sum_j e^{x_j - m_s} V_j
 * (x_j = scale * q . K_j, natural-log units), and a combine kernel merges them
 * with one global 1/l_g.
 *
 *   q [B,H,1,D]                    input, dtype
 *   Kcache, Vcache [B,H,N,D]       input, dtype
 *   O [B,H,1,D]                    output, dtype
 *   partial_ws                     caller-owned scratch of
 *                                  fa_decode_workspace_bytes(B,H,D,n_splits)
 *                                  bytes; on return it holds, float32,
 *                                  O_s [B*H][n_splits][D], then m_s
 *                                  [B*H][n_splits], then l_s [B*H][n_splits]
 *                                  (an empty split has m_s = -inf, l_s = 0)
 *   scale                          any finite value
 *   n_splits                       1 <= n_splits <= min(N, 65535); B*H <= 65535
 */
fa_status fa_decode(const void* q, const void* Kcache, const void* Vcache, void* O, float* partial_ws, int B,
                    int H, int N, int D, float scale, int n_splits, fa_dtype dtype, void* stream);

/* Bytes of scratch fa_decode needs: B*H*n_splits*(D+2) float32. */
size_t fa_decode_workspace_bytes(int B, int H, int D, int n_splits);

/*
 * Decode of R query rows per (batch, head), with an optional LSE.
 *
 * The same split-and-combine as fa_decode, for R >= 1 query rows that all see
 * the whole cache of their (batch, head) (no mask among them): for example the
 * R query heads of grouped-query attention that share one K/V head, laid out
 * as that head's rows. Each K and V vector read from HBM serves all R rows.
 * fa_decode is this call with R = 1 and LSE = NULL.
 *
 *   q [B,H,R,D]                    input, dtype
 *   Kcache, Vcache [B,H,N,D]       input, dtype
 *   O [B,H,R,D]                    output, dtype
 *   LSE [B,H,R]                    output, float32, natural log of the row's
 *                                  softmax denominator over scaled scores
 *                                  (m_g + ln l_g), or NULL for none
 *   partial_ws                     caller-owned scratch of
 *                                  fa_decode_ex_workspace_bytes(B,H,R,D,n_splits)
 *                                  bytes; on return, float32, O_s
 *                                  [B*H*R][n_splits][D], then m_s
 *                                  [B*H*R][n_splits], then l_s, row
 *                                  (b*H + h)*R + r
 *   R                              1 <= R <= 4; R > 4 is FA_ERR_UNSUPPORTED
 *                                  (fa_fwd with M = R takes any number of rows)
 *   scale, n_splits                as for fa_decode
 */
fa_status fa_decode_ex(const void* q, const void* Kcache, const void* Vcache, void* O, float* LSE,
                       float* partial_ws, int B, int H, int R, int N, int D, float scale, int n_splits,
                       fa_dtype dtype, void* stream);

/* Bytes of scratch fa_decode_ex needs: B*H*R*n_splits*(D+2) float32. */
size_t fa_decode_ex_workspace_bytes(int B, int H, int R, int D, int n_splits);

/*
 * Decode that allocates nothing and needs no workspace argument.
 *
 * The pages have no counterpart to this call; it exists for callers that
 * cannot allocate device memory when they decode (a caching or arena allocator
 * that must not grow, a runtime that accounts for every buffer itself, a C
 * caller without an allocator at hand). Same arguments, layouts and result as
 * fa_decode, minus partial_ws: the split partials go to a fixed 16 MiB float32
 * array inside the library's device image, which every GPU that loads the
 * library holds until the process exits.
 *
 * - Limit: B*H*n_splits*(D+2) <= 4,194,304 floats (e.g. B=8, H=32, D=128 with
 *   up to 126 splits); larger requests return FA_ERR_INVALID, naming the limit,
 *   and launch nothing.
 * - The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture on the device.
 * - Calls, cudaMalloc and cudaFree: none. The array is shared by every call on
 *   a device and keeps the last call's partials. Nothing in it needs to start
 *   at zero (each call writes every partial it reads), but calls that overlap
 *   on the GPU (e.g. on two streams at once) race on it: serialise them.
 */
fa_status fa_decode_static(const void* q, const void* Kcache, const void* Vcache, void* O, int B, int H, int N,
                           int D, float scale, int n_splits, fa_dtype dtype, void* stream);

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * word. FA_ERR_TIMEOUT if a kernel gave up a bounded wait since the last call
 * (fa_last_error_message() names the kernel and the wait), FA_ERR_CUDA if the
 * synchronisation itself failed, FA_OK otherwise. The status word is shared by
 * all streams of a device.
 */
fa_status fa_last_status(void* stream);

/* Static string for a status code. */
const char* fa_status_string(fa_status s);

/* One-line description of the last error on the calling host thread. */
const char* fa_last_error_message(void);

/*
 * Bound, in nanoseconds, on every wait inside the kernels launched by this
 * library after the call (default 2e9, i.e. 2 s; the environment variable
 * FA_WAIT_BUDGET_NS overrides the default at first use). Values < 1000 are
 * FA_ERR_INVALID.
 */
fa_status fa_set_wait_budget_ns(unsigned long long ns);

/*
 * Schedule controls (no counterpart on the pages). The library chooses some
 * work schedules per call from the problem's shape; these fix a choice instead,
 * for tuning and for tests that must reach each schedule. Process-wide (every
 * device, every thread); results do not depend on them beyond the f32 summation
 * order the split schedules document. value -1 restores the automatic choice,
 * which is the default.
 *   FA_SCHED_FWD_SPLIT    0 / 1: the D = 64 forward's split schedule (fa_fwd_ws,
 *                         fa_fwd_host) off / on
 *   FA_SCHED_BWD_SPLIT    0 / 1: the fused backward's split schedule (fa_bwd_ws,
 *                         non-causal, D = 64) off / on
 *   FA_SCHED_HOST_CHUNKS  1..8: number of equal head chunks fa_fwd_host
 *                         pipelines (default -1: three chunks, 4:2:1;
 *                         fa_fwd_host_workspace_bytes depends on it)
 *   FA_SCHED_BWD_PAIR     0 / 1: fa_bwd's dK/dV and dQ kernels (D = 64) on CTA
 *                         pairs (tcgen05 cta_group::2, 256 rows per pair) off / on;
 *                         automatic: on for non-causal calls with fewer key
 *                         tiles than SMs
 * Other keys or values: FA_ERR_INVALID.
 */
typedef enum fa_sched_key {
  FA_SCHED_FWD_SPLIT = 1,
  FA_SCHED_BWD_SPLIT = 2,
  FA_SCHED_HOST_CHUNKS = 3,
  FA_SCHED_BWD_PAIR = 4
} fa_sched_key;
fa_status fa_set_schedule(fa_sched_key key, int value);

/*
 * Test-only fault injection (no counterpart on the pages; exercises the bounded
 * waits described at fa_set_wait_budget_ns). One-shot: the next launch of the
 * kind named consumes it; kind 0 cancels a pending injection; other kinds are
 * FA_ERR_INVALID. In each case a bounded wait runs out, the CTAs drain and exit,
 * and fa_last_status reports FA_ERR_TIMEOUT naming the kernel and the wait site;
 * nothing faults and the context stays usable.
 *   1  next fa_decode / fa_decode_static launch: its first CTA never loads its
 *      first stage of keys (a wait inside one CTA)
 *   2  next fp16/bf16 D = 64 forward: its first CTA never loads its first stage
 *      of K/V (waits inside one CTA)
 *   3  next fp16/bf16 D = 64 forward on the split schedule: CTA 1 never
 *      publishes the partial of its first piece, so the CTA that merges it
 *      gives up its wait on CTA 1's flags (a wait between CTAs)
 *   4  next fa_bwd_ws call on the fused pass's split schedule: the lowest CTA
 *      whose share starts inside a key tile never counts its partial in, so
 *      the CTA holding that tile's first query blocks gives up its wait for
 *      the count (a wait between CTAs)
 */
fa_status fa_debug_inject(int kind);

/*
 * Test-only: the schedule the library would choose, without launching anything
 * (no GPU needed). which = 0: the fp16/bf16 D = 64 forward with a workspace
 * (fa_fwd_ws); which = 1: the fused backward (fa_bwd_ws, D = 64). num_sms is
 * the device's SM count to assume. Returns 1 for the split schedule, 0 for
 * whole query pairs / key tiles, -1 for an unknown `which` or a non-positive
 * size. A setting made with fa_set_schedule applies as it does to the calls.
 */
int fa_debug_schedule_choice(int which, int B, int H, int M, int N, int causal, int num_sms);

#ifdef __cplusplus
}
#endif

#endif /* FA_H */
