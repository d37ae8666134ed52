/*
 * jfa.h -- C ABI of libjfa.so: Jagged Flash Attention forward and backward
 * for NVIDIA GB300 (sm_103a).
 *
 * The operation.  Sequences of different lengths are packed back to back
 * with no padding, and an int32 offsets tensor records where each one
 * starts; FlashAttention runs directly on the packed Q/K/V ("Why attention
 * in GEM needed a rewrite", Meta's TLX Jagged Flash Attention Beats FA4 on
 * Blackwell With 3x Less Code; Meta's 3.2K-line Triton kernel outruns
 * FlashAttention-4 on jagged Blackwell attention, third paragraph).  For
 * sequence b (keys offsets[b] .. offsets[b+1]-1) and head h:
 *
 *     S = scale * Q K^T,  P = softmax(S) row-wise,  O = P V,
 *     LSE = natural log of the row sums of exp(S).
 *
 * Two query modes:
 *   broadcast_q = 1: one dense Q [Lq,H,D] is shared by every sequence, and
 *     dQ is the sum over the whole batch of each sequence's gradient (Meta's
 *     3.2K-line Triton kernel ..., second paragraph; Meta's TLX Jagged Flash
 *     Attention ..., section "Optimizations layered on top").
 *   broadcast_q = 0: jagged self-attention; Q is packed like K/V and
 *     sequence b's queries are rows offsets[b] .. offsets[b+1]-1.  `causal`
 *     (query i sees keys j <= i, counted from the sequence start) is only
 *     defined in this mode.
 *
 * Layouts (all row-major, contiguous, device memory):
 *   q    bf16  [Lq, H, D] (broadcast) or [N, H, D] (jagged), N = offsets[B]
 *   k, v bf16  [N, H, D]
 *   o    bf16  [B, Lq, H, D] (broadcast) or [N, H, D]
 *   lse  fp32  [B, H, Lq]    (broadcast) or [H, N]
 *   dout bf16  shaped like o
 *   dq   fp32  shaped like q (the library zeroes it before accumulating)
 *   dk, dv bf16 [N, H, D]
 * Empty sequences are allowed: their O rows are 0, their LSE is -inf and
 * they add nothing to dQ.
 *
 * Supported: D in {64, 128}; 1 <= H <= 255; every sequence no longer than
 * 2^23 rows; N < 2^31; broadcast Lq <= 2^23.  Arithmetic: bf16 operands on
 * the tensor cores with fp32 accumulation; softmax statistics in fp32.
 *
 * Ownership and concurrency.  The caller owns every device buffer and the
 * stream.  The library allocates no device memory; it keeps a small pinned
 * host staging ring per device for the tile schedule: the plain forward's
 * kernel reads its work list there through the ring's device mapping, the
 * dense backward's Delta pass moves it into the workspace the same way, and
 * the other paths (block-sparse, MXFP8, split-KV tables) copy it into the
 * workspace; where the ring is not mapped, it is copied.  Scratch memory (the
 * tile schedule, the backward row statistics and a status word) lives in the
 * caller's `workspace`, which must hold jfa_workspace_bytes(...) bytes and
 * must not be shared by calls that may run concurrently.  Calls are
 * asynchronous on `stream`; the one exception is that, when offsets_host is
 * NULL, the library first copies the offsets from the device synchronously.
 *
 * Errors are returned, never thrown.  A call that returns anything but
 * JFA_OK has enqueued no work, except JFA_ERR_CUDA, which reports a failed
 * launch.  Kernels never trap: a bounded wait that times out records
 * JFA_ERR_DEVICE_TIMEOUT in the workspace, which jfa_device_status() reads.
 */
#ifndef JFA_H
#define JFA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    JFA_OK = 0,
    JFA_ERR_INVALID_ARG = 1,   /* null pointer, negative size, bad offsets, non-finite scale */
    JFA_ERR_UNSUPPORTED = 2,   /* D not in {64,128}, causal with broadcast_q, misaligned pointer, size limits */
    JFA_ERR_WORKSPACE = 3,     /* workspace missing, misaligned or smaller than jfa_workspace_bytes() */
    JFA_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed */
    JFA_ERR_DEVICE_TIMEOUT = 5 /* a kernel's bounded wait expired (reported by jfa_device_status) */
} jfa_status;

/*
 * Bytes of workspace one call needs (forward or backward) for a batch of B
 * sequences holding total_len = offsets[B] rows in all, Lq broadcast query
 * rows (ignored when broadcast_q == 0), H heads and head dimension D.  The
 * same workspace serves jfa_fwd and jfa_bwd.  Returns 0 for unsupported or
 * invalid sizes.  The workspace must be 256-byte aligned.
 */
size_t jfa_workspace_bytes(int B, int total_len, int Lq, int H, int D, int broadcast_q, int causal);

/*
 * jfa_fwd -- O and LSE (the forward pass).
 *   q, k, v      device bf16 inputs (layouts above), 16-byte aligned.
 *   offsets_dev  device int32 [B+1]; may be NULL when offsets_host is given.
 *   offsets_host host int32 [B+1]; may be NULL (then copied from offsets_dev,
 *                synchronously).  offsets[0] must be 0 and offsets must not
 *                decrease.
 *   scale        softmax scale; <= 0 selects 1/sqrt(D).
 *   o, lse       device outputs (layouts above).
 *   workspace    device scratch of at least jfa_workspace_bytes() bytes.
 *   stream       cudaStream_t (NULL = legacy default stream).
 * Load balance: the host deals (sequence, head, query-tile) items to one
 * persistent CTA per SM, longest first.  In broadcast mode a query tile
 * whose key loop alone costs more than 1.5x an average CTA's share is split into
 * key chunks (split-KV); each chunk writes an fp32 partial O and LSE into
 * the workspace (at most 512 chunks per call) and a merge kernel combines
 * them (LSE = ln sum_c exp(LSE_c), O = sum_c exp(LSE_c - LSE) O_c).
 */
jfa_status jfa_fwd(const void *q, const void *k, const void *v, const int32_t *offsets_dev,
                   const int32_t *offsets_host, int B, int Lq, int H, int D, int broadcast_q, int causal,
                   float scale, void *o, float *lse, void *workspace, size_t workspace_bytes, void *stream);

/*
 * jfa_bwd -- dQ, dK, dV (the backward pass) given the forward's O and LSE
 * and the upstream gradient dout.  A first kernel computes Delta =
 * rowsum(dout * o) into the workspace, then the main kernel runs.  dq is
 * fp32 and is overwritten
 * (zeroed, then summed over every sequence in broadcast mode); dk and dv are
 * bf16.  Other arguments as for jfa_fwd.  dQ is accumulated with fp32
 * atomics, so its low-order bits may differ from run to run; dK and dV are
 * deterministic.
 */
jfa_status jfa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
                   const void *dout, const int32_t *offsets_dev, const int32_t *offsets_host, int B, int Lq, int H,
                   int D, int broadcast_q, int causal, float scale, float *dq, void *dk, void *dv, void *workspace,
                   size_t workspace_bytes, void *stream);

/*
 * Block-sparse variant: attention restricted to selected blocks of keys.
 * The pages' block-sparse kernel only adds iteration over selected blocks
 * and leaves the rest unchanged (TLX porta l'attenzione jagged su Blackwell
 * oltre FA4 con un terzo del codice, section "The turning point").  Keys
 * come in blocks of 128 counted from each sequence's start (the last block of
 * a sequence may be shorter); a selection applies to a (sequence, head) pair
 * as a whole, i.e. to every query row of that sequence and head:
 *
 *   kv_block_mask  HOST uint8 [NB, H], row-major, NB = jfa_num_kv_blocks():
 *                  entry (block_start[b] + n) * H + h != 0 selects key
 *                  block n of sequence b for head h, where block_start[b] =
 *                  sum over b' < b of ceil(len_b' / 128).  Read during the
 *                  call only (the selection is turned into the tile schedule
 *                  on the host); the caller keeps ownership.
 *
 * Keys of unselected blocks are treated like keys outside the sequence: they
 * get no weight, and their dK and dV rows are written as zeros.  A query row
 * whose (sequence, head) selects no block gets O = 0, LSE = -inf and adds
 * nothing to dQ.  Work scales with the selected blocks.  Not defined with
 * causal masking (there is no causal argument).  All other arguments,
 * layouts, the workspace (jfa_workspace_bytes() covers it) and the error
 * behaviour are those of jfa_fwd / jfa_bwd; a NULL mask returns
 * JFA_ERR_INVALID_ARG.
 */
jfa_status jfa_fwd_block_sparse(const void *q, const void *k, const void *v, const int32_t *offsets_dev,
                                const int32_t *offsets_host, const uint8_t *kv_block_mask, int B, int Lq, int H,
                                int D, int broadcast_q, float scale, void *o, float *lse, void *workspace,
                                size_t workspace_bytes, void *stream);
jfa_status jfa_bwd_block_sparse(const void *q, const void *k, const void *v, const void *o, const float *lse,
                                const void *dout, const int32_t *offsets_dev, const int32_t *offsets_host,
                                const uint8_t *kv_block_mask, int B, int Lq, int H, int D, int broadcast_q,
                                float scale, float *dq, void *dk, void *dv, void *workspace, size_t workspace_bytes,
                                void *stream);

/*
 * MXFP8 variant of the forward.  The pages' MXFP8 kernel runs its matmuls in
 * microscaling precision, quantizing P to FP8 on the fly and keeping the
 * scale factors in tensor memory (TLX porta l'attenzione jagged su Blackwell
 * oltre FA4 con un terzo del codice, section "The turning point").  Here the
 * P V product is MXFP8 (E4M3 elements, one E8M0 scale 2^(code - 127) per 32
 * elements along the keys); Q K^T stays bf16.
 *
 *   v8       device uint8 [N, H, D]: V as E4M3 codes (1 sign, 4 exponent
 *            bits with bias 7, 3 mantissa bits; S.1111.111 is NaN).
 *   v_scale  device uint8 [NB, H, D, 4], NB = jfa_num_kv_blocks(), 16-byte
 *            aligned: byte [block_start[b] + n][h][d][c] is the scale code of
 *            keys 128 n + 32 c .. + 31 of sequence b in column d (block_start
 *            as for the block-sparse mask).  jfa_quantize_v_mxfp8 writes both.
 *
 * P is quantized per row and 32-key chunk c (counted from the sequence
 * start): with x = scale * s * log2(e), X_c = floor(max_c x) - 8 and the
 * weight 2^x becomes 2^X_c * E4M3(2^(x - X_c)) (nearest, ties to even,
 * saturating at 448).  O = sum_j pq_j v_j / sum_j 2^(x_j): the normaliser is
 * the row sum of the unquantized weights, and LSE is the bf16 forward's.
 * Split-KV is not used.  All other arguments, layouts, the workspace and the
 * errors are those of jfa_fwd; a NULL v_scale with N > 0 returns
 * JFA_ERR_INVALID_ARG.
 */
jfa_status jfa_fwd_mxfp8(const void *q, const void *k, const void *v8, const void *v_scale,
                         const int32_t *offsets_dev, const int32_t *offsets_host, int B, int Lq, int H, int D,
                         int broadcast_q, int causal, float scale, void *o, float *lse, void *workspace,
                         size_t workspace_bytes, void *stream);

/*
 * jfa_quantize_v_mxfp8 -- MXFP8 V for jfa_fwd_mxfp8 from bf16 v [N, H, D].
 * Per sequence b, 128-key block n, head h, column d and 32-key chunk c:
 * X = floor(log2(max |v|)) - 8 over the chunk's keys (clamped to [-127, 127];
 * -127 for an all-zero chunk), v8 = E4M3(v / 2^X) for those keys, and scale
 * code X + 127; chunks past the sequence end get code 0.  Exact: the codes
 * do not depend on rounding order.  offsets_dev is required (the kernel reads
 * it); offsets_host as for jfa_fwd.  workspace: 256-byte aligned, at least
 * 256 + 4 (B + 1) bytes (any jfa_workspace_bytes() workspace of the same B
 * qualifies).  v, v8 and v_scale must be 16-byte aligned.
 */
jfa_status jfa_quantize_v_mxfp8(const void *v, const int32_t *offsets_dev, const int32_t *offsets_host, int B,
                                int H, int D, void *v8, void *v_scale, void *workspace, size_t workspace_bytes,
                                void *stream);

/* NB = sum over the B sequences of ceil(len_b / 128) (host offsets [B+1]); -1 for bad arguments. */
int64_t jfa_num_kv_blocks(const int32_t *offsets_host, int B);

/*
 * jfa_device_status -- synchronises `stream`, then reads and clears the
 * status word kernels write into `workspace`.  Returns JFA_OK,
 * JFA_ERR_DEVICE_TIMEOUT, or JFA_ERR_CUDA if the synchronisation failed.
 */
jfa_status jfa_device_status(void *workspace, void *stream);

/*
 * jfa_set_wait_limit -- how long one barrier wait inside the kernels may
 * last before the kernel gives up (process-wide, for launches after the
 * call; 0 restores the default of 4 s).  A wait that runs out sets the
 * status word (JFA_ERR_DEVICE_TIMEOUT through jfa_device_status), makes the
 * CTA's other waits give up, lets the CTA's issued copies and products
 * finish, frees its tensor memory and returns; the outputs are then
 * incomplete.  Legitimate waits last microseconds.
 */
jfa_status jfa_set_wait_limit(unsigned long long ns);

/* Static, human-readable name of a status code. */
const char *jfa_status_string(jfa_status s);

/*
 * jfa_fwd_static_scratch -- jfa_fwd for callers that cannot allocate memory.
 * The pages describe no such entry point; it exists for code that cannot
 * provide a workspace, such as a plugin inside an engine that owns all device
 * memory and forbids allocation while it runs, or a program restricted to a
 * fixed memory pool.  It computes exactly what jfa_fwd computes, with the
 * same arguments minus the workspace; offsets_host is required.
 *
 * Scratch (tile schedule and status word) lives in a 1 MiB array the library
 * declares in device global memory; every GPU that loads the library holds
 * it until the process exits.  The call makes no allocation of any kind (no
 * cudaMalloc/cudaFree, no pinned or heap memory).  Limit: at most 65,264
 * forward work items (H x the number of 256-row query-tile pairs summed over
 * the sequences); larger batches return JFA_ERR_WORKSPACE before any work is
 * enqueued.  Every call shares the array and overwrites what the previous
 * call left there; calls whose work overlaps on the GPU (other streams or
 * threads) race on it and must be serialised by the caller.  The first call
 * on each device looks up the array's device address (cudaGetSymbolAddress)
 * and keeps it for the rest of the process, so the entry point does not
 * survive cudaDeviceReset; make that first call before any stream capture.
 * The schedule is copied into the array from a host buffer that each call
 * rewrites, so a call on a stream that is capturing returns
 * JFA_ERR_UNSUPPORTED and enqueues nothing.  A kernel wait that times out is
 * recorded in the array's status word, which each call clears at its start;
 * jfa_static_scratch_status() reports it.
 */
jfa_status jfa_fwd_static_scratch(const void *q, const void *k, const void *v, const int32_t *offsets_host, int B,
                                  int Lq, int H, int D, int broadcast_q, int causal, float scale, void *o, float *lse,
                                  void *stream);

/*
 * jfa_static_scratch_status -- synchronises `stream`, then reads and clears
 * the status word of jfa_fwd_static_scratch's array on the current device.
 * Returns JFA_OK, JFA_ERR_DEVICE_TIMEOUT, or JFA_ERR_CUDA if the
 * synchronisation or the read failed.  Like that entry point, it allocates
 * nothing.
 */
jfa_status jfa_static_scratch_status(void *stream);

/*
 * Measurement aid (computes nothing).  While enabled, every forward and
 * backward call also records a pair of CUDA events on its stream around each
 * of the library's kernels.  jfa_profile_read() waits for the recorded
 * events and writes, for kernel kind k < count, the summed milliseconds into
 * ms[k] and the launch count into launches[k] (either pointer may be NULL),
 * then clears the totals.  Kinds: 0 forward kernel, 1 backward Delta
 * pre-pass, 2 backward main kernel, 3 block-sparse zeroing of unselected
 * dK/dV tiles, 4 split-KV merge, 5 MXFP8 quantization of V.  The events
 * are host-owned CUDA events; no device memory is allocated.
 */
jfa_status jfa_profile_enable(int on);
jfa_status jfa_profile_read(double *ms, int *launches, int count);

/*
 * jfa_set_schedule_policy -- measurement aid: how later calls deal their
 * sorted work items to the persistent CTAs (process-wide, all devices).
 * 0 = longest first, zigzag over the CTAs (the pages' deal: Meta's TLX
 * Jagged Flash Attention Beats FA4 on Blackwell With 3x Less Code, section
 * "Optimizations layered on top"); 1 = generation order, round-robin (no
 * balancing); 2 = longest first, each item to the least-loaded CTA.
 * Backward only: 3 = Cluster Launch Control (the pages list it among the
 * primitives that keep SMs busy under length skew: same page, sections "What
 * TLX changes" and "Optimizations layered on top"): the longest-first list,
 * one CTA per item, and every resident CTA, when it starts an item, asks the
 * hardware to cancel a CTA that has not started yet and takes over its item
 * -- a deal made at run time by whichever SM is free; 4 = queues: one CTA
 * per SM as in the static deals, the items of each head group (broadcast Q
 * with H dividing the CTA count; otherwise all items) in one longest-first
 * queue, and each CTA, as it starts an item, atomically takes the next item
 * of its group's queue -- a run-time deal that keeps each CTA on one head.
 * Defaults: 2 for the forward, 0 for the backward.  Results do not depend on
 * the policy (up to dQ's summation order); only the time does.  Returns
 * JFA_ERR_INVALID_ARG for another value.
 */
jfa_status jfa_set_schedule_policy(int fwd_policy, int bwd_policy);

/*
 * jfa_num_ctas -- number of persistent CTAs the kernels launch on the current
 * device (one per SM); the schedule deals work to exactly this many.
 */
int jfa_num_ctas(void);

#ifdef __cplusplus
}
#endif
#endif /* JFA_H */
