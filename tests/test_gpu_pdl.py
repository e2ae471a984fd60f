"""Back-to-back GEMMs launched as programmatic dependents (LCGEMM_OPT_PDL): each kernel may start its
prologue while the one before it runs, but reads and writes global memory only after it completed.
Checked on every plain kernel, with the option on and off: a GEMM whose A is the previous GEMM's
output (read after write; that output starts as NaN) and two GEMMs writing the same C (write after
write)."""
import pytest
import torch

import complexity_matmul_gb300 as lcg
import synthetic
from helpers import assert_bit_exact, assert_close, oracle_c64

pytestmark = pytest.mark.gpu

# (plain kernel option, M, N1, K, N2): CTA-pair tiles; single-CTA tiles with 3 K chunks summed by
# the last to arrive; single-CTA tiles with 8 chunks summed by the reduction kernel; the stream-K
# skinny kernel; the GEMV
CASES = [(2, 512, 512, 64, 256), (1, 100, 384, 3072, 200), (1, 40, 128, 8192, 64), (3, 16, 1024, 256, 512),
         (4, 1, 1024, 512, 2048)]


def _handle(kernel, pdl):
    h = lcg.Handle(0)
    h.set_option(lcg.OPT_PLAIN_KERNEL, kernel)
    h.set_option(lcg.OPT_PDL, pdl)
    return h


@pytest.mark.parametrize("pdl", [1, 0])
@pytest.mark.parametrize("kernel,M,N1,K,N2", CASES)
def test_read_after_write(kernel, M, N1, K, N2, pdl):
    h = _handle(kernel, pdl)
    A, B = synthetic.operands(M, N1, K, "int3", 95, "bf16", "cuda")
    D = synthetic.matrix(N2, N1, "int3", 96, "bf16", "cuda")
    C1 = torch.full((M, N1), float("nan"), dtype=torch.bfloat16, device="cuda")
    C2 = torch.empty((M, N2), dtype=torch.bfloat16, device="cuda")
    for _ in range(3):
        h.run(A, B, C1, algo="plain")
        h.run(C1, D, C2, algo="plain")       # A of this GEMM is the output of the one before
    torch.cuda.synchronize()
    assert h.sync_status() == 0
    assert_bit_exact(C1, oracle_c64(A, B, "bf16"), "bf16")
    assert not torch.isnan(C2.float()).any()
    assert_close(C2, oracle_c64(C1, D, "bf16"), "bf16", "plain")
    h.close()


@pytest.mark.parametrize("pdl", [1, 0])
@pytest.mark.parametrize("kernel,M,N1,K,N2", CASES)
def test_write_after_write(kernel, M, N1, K, N2, pdl):
    h = _handle(kernel, pdl)
    A1, B1 = synthetic.operands(M, N1, K, "int3", 97, "bf16", "cuda")
    A2, B2 = synthetic.operands(M, N1, K, "int3", 98, "bf16", "cuda")
    C = torch.empty((M, N1), dtype=torch.bfloat16, device="cuda")
    for _ in range(3):
        h.run(A1, B1, C, algo="plain")
        h.run(A2, B2, C, algo="plain")       # the later GEMM's values must be the ones left in C
    torch.cuda.synchronize()
    assert h.sync_status() == 0
    assert_bit_exact(C, oracle_c64(A2, B2, "bf16"), "bf16")
    h.close()
