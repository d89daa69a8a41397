"""Failure path of the kernels' bounded waits on the GPU, without a fault: a
wait that nothing satisfies gives up after its limit, raises TSA_FLAG_TIMEOUT
for the host to read, and leaves the CUDA context usable."""
import time

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tsa():
    import trainable_sparse_attention_gb300 as m
    m.build()
    m.load_library()
    return m


def test_bounded_wait_gives_up_and_the_context_survives(tsa):
    tsa.read_flags(clear=True)
    t0 = time.perf_counter()
    tsa.selftest_bounded_wait()
    flags = tsa.read_flags(clear=True)  # synchronises the stream
    waited = time.perf_counter() - t0
    assert flags & tsa.FLAG_TIMEOUT
    assert waited >= 1.5  # the wait ran out its 2 s limit rather than passing early
    # later launches on the same context still compute correctly
    x = torch.randn(4, 300, device="cuda")
    got = tsa.qsa_topk_from_scores(x, 5)
    assert torch.equal(got.long(), torch.topk(x, 5, dim=-1).indices)
    assert tsa.read_flags() == 0
