"""Runs after the other GPU tests of the session (file order): none of the
bounded pipeline waits (TMA-streamed GEMV, tensor-core GEMM) ran out while
they ran.  A wait that runs out lets its kernel finish with wrong numbers and
counts itself here instead of hanging the GPU."""
import pytest


@pytest.fixture(scope="module")
def sub():
    import substitute_speculative_decoding_gb300 as s
    return s


@pytest.mark.gpu
def test_no_pipeline_wait_ran_out(sub):
    import torch
    torch.cuda.synchronize()
    assert sub.pipeline_timeouts() == 0
