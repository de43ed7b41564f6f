"""Failure detection without a GPU fault: a wait inside the tensor-core kernel
that can never complete (one operand stage is never announced) must give up
after its time limit, raise KD_FLAG_TIMEOUT, stop both CTAs of every pair, and
leave the context usable -- the next GEMM on the same stream is correct."""
import time

import pytest

pytestmark = pytest.mark.gpu


def test_withheld_arrival_times_out_and_the_context_survives(kd):
    import torch
    lib = kd.load_library()
    g = torch.Generator().manual_seed(3)
    M, N, K = 512, 512, 256
    A = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    B = torch.randn(N, K, generator=g).to(torch.bfloat16).cuda()
    D = torch.zeros(M, N, dtype=torch.float32, device="cuda")
    counter = torch.zeros(1, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    st = lib.kd_umma_gemm_bf16_wait_test(A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K,
                                         20000, counter.data_ptr(), err.data_ptr(),
                                         torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(err.item()) & kd.KD_FLAG_TIMEOUT
    assert elapsed < 3.0, elapsed   # 20 ms limit, plus the fixed drain of in-flight copies
    # the same stream and context still compute correctly
    out, err2 = kd.kd_umma_gemm_bf16(A, B, M, N, K, False, False)
    torch.cuda.synchronize()
    assert int(err2.item()) == 0
    want = A.double() @ B.double().T
    assert float((out.cpu().double() - want.cpu()).abs().max()) <= 2e-5 * float(want.abs().max()) + 1e-4
