"""The sm_103a rule that rules out a CTA-pair (2-CTA) backward of this design.

The pages' last backward optimisation lets two CTAs cooperate on one matmul
(Meta's TLX Jagged Flash Attention Beats FA4 on Blackwell With 3x Less Code,
section "Optimizations layered on top").  On sm_103a that is tcgen05 with
`.cta_group::2`, and ptxas does not let one kernel use both `.cta_group::1`
and `.cta_group::2`.  A pair of CTAs on two key tiles of one (sequence, head)
can express S^T, dP^T, dV and dK as pair products (their B operands, Q and
dO, are shared), but dQ = dS K sums over the pair's keys with a different K
in each CTA, so it has no pair form; pairing two query tiles instead leaves
dK and dV (sums over the pair's queries) without one.  This test compiles the
two cases with the toolkit's nvcc (no GPU needed): a kernel mixing the two
granularities is rejected, the same kernel with pair operations only builds.
"""
import os
import shutil
import subprocess

import pytest

NVCC = shutil.which("nvcc") or ("/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else None)

KERNEL = r"""
#include <cstdint>
__global__ void __cluster_dims__(2, 1, 1) k(uint32_t* out, uint64_t adesc, uint64_t bdesc) {
    __shared__ uint32_t tbase;
    __shared__ uint64_t bar;
    const uint32_t bar_a = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
    if (threadIdx.x < 32)
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], 256;"
                     ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(&tbase))));
    __syncthreads();
    const uint32_t t = tbase;
    if (threadIdx.x == 0) {
        asm volatile("{.reg .pred p; setp.ne.b32 p, %3, 0; tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;}"
                     ::"r"(t), "l"(adesc), "l"(bdesc), "r"(0u));
        SECOND_PRODUCT
        asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
                     ::"r"(bar_a), "h"(static_cast<uint16_t>(3)));
    }
    __syncthreads();
    if (threadIdx.x < 32) asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, 256;" ::"r"(t));
    out[threadIdx.x] = t;
}
"""
SINGLE = ('asm volatile("{.reg .pred p; setp.ne.b32 p, %3, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;}"'
          '::"r"(t + 128), "l"(adesc), "l"(bdesc), "r"(0u));')
PAIR = ('asm volatile("{.reg .pred p; setp.ne.b32 p, %3, 0; tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;}"'
        '::"r"(t + 128), "l"(adesc), "l"(bdesc), "r"(0u));')


def _compile(tmp_path, second):
    src = tmp_path / "pair.cu"
    src.write_text(KERNEL.replace("SECOND_PRODUCT", second))
    return subprocess.run([NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-c", str(src), "-o",
                           str(tmp_path / "pair.o")], capture_output=True, text=True)


@pytest.mark.skipif(NVCC is None, reason="needs the CUDA toolkit's nvcc")
def test_single_and_pair_products_do_not_mix(tmp_path):
    mixed = _compile(tmp_path, SINGLE)
    assert mixed.returncode != 0
    assert "cta_group" in (mixed.stdout + mixed.stderr)
    pair_only = _compile(tmp_path, PAIR)
    assert pair_only.returncode == 0, pair_only.stderr
