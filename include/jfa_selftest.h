/*
 * jfa_selftest.h -- diagnostic entry point of libjfa.so (not part of the
 * attention path).
 *
 * The attention kernels stage operands with TMA into 128-byte-swizzled
 * shared memory and multiply them on the tcgen05 tensor cores into TMEM.
 * This entry point runs exactly one such 128x128x128 bf16 product so a test
 * can check the operand descriptors against a library matmul on the GPU.
 * The pages describe the kernel's use of "async TMA and MMA" and "explicit
 * SMEM and TMEM allocation" (Meta's 3.2K-line Triton kernel outruns
 * FlashAttention-4 on jagged Blackwell attention, last paragraph); this
 * checks our own sm_103a realisation of those primitives.
 */
#ifndef JFA_SELFTEST_H
#define JFA_SELFTEST_H

#ifdef __cplusplus
extern "C" {
#endif

/*
 * jfa_selftest_mma -- C (fp32, [128][128] row-major, device) from bf16
 * device matrices a and b (each [128][128] row-major, 16-byte aligned):
 *   mode 0: C = A  B^T   (A [M][K], B [N][K], both K-major)
 *   mode 1: C = A  B     (A [M][K] K-major, B [K][N] MN-major)
 *   mode 2: C = A  B     (as mode 1, A staged through tensor memory)
 *   mode 3: C = A^T B    (A given as [K][M], B as [K][N], both MN-major)
 *   mode 4: C = A  B     (as mode 1, issued as two N=64 halves)
 * status: device uint32, OR-ed with a nonzero bit if a wait timed out.
 * Asynchronous on `stream` (a cudaStream_t).  Returns 0 on launch, 1 on a
 * bad argument, 4 on a CUDA error.  Allocates nothing.
 */
int jfa_selftest_mma(int mode, const void *a, const void *b, float *c, unsigned int *status, void *stream);

/*
 * jfa_selftest_timeout -- exercises the kernels' failure path without a
 * fault: one CTA whose warp 1 waits on a barrier nothing ever completes,
 * bounded by limit_ns (1 ns .. 1 s), and whose warp 2 waits the same way
 * with a limit 2000 times longer, so it returns early only if the CTA abort
 * flag that warp 1's timeout raises reaches it.  The CTA also holds tensor
 * memory, which it frees before returning.  On return, *status (device
 * uint32) has the timeout bit set and out[0..1] (device uint32) are 0 for
 * each warp that gave up.  Asynchronous on `stream`.  Returns 0 on launch,
 * 1 on a bad argument, 4 on a CUDA error.  Allocates nothing.
 */
int jfa_selftest_timeout(unsigned long long limit_ns, unsigned int *status, unsigned int *out, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* JFA_SELFTEST_H */
