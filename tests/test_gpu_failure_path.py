"""The failure path of the bounded in-kernel waits, exercised without a fault:
q4k_selftest_timeout launches a one-thread kernel whose wait on an mbarrier that
nothing arrives at runs out after a short limit. The device error word must
then read Q4K_ERR_TIMEOUT, clearing it must work, and the context must stay
usable: a matmul right after it is clean and correct."""
import numpy as np
import pytest
import torch

from gguf_q4_dequant_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(autouse=True)
def _cuda(q4k):
    if not torch.cuda.is_available():
        pytest.fail("GPU tests need a CUDA device")
    torch.cuda.set_device(0)
    q4k.q4k_init()
    assert q4k.q4k_device_error(clear=True) in (0, q4k.Q4K_ERR_TIMEOUT)
    yield
    torch.cuda.synchronize()
    q4k.q4k_device_error(clear=True)


@pytest.mark.parametrize("limit_ns", [1_000, 1_000_000])
def test_timed_out_wait_sets_the_error_word(q4k, oracle_mod, limit_ns):
    q4k.q4k_selftest_timeout(limit_ns)
    torch.cuda.synchronize()
    assert q4k.q4k_device_error(clear=False) == q4k.Q4K_ERR_TIMEOUT
    assert q4k.q4k_device_error(clear=True) == q4k.Q4K_ERR_TIMEOUT  # reads, then clears
    assert q4k.q4k_device_error(clear=False) == 0

    # the context is intact: a normal call afterwards leaves the word clean and is correct
    N, K = 300, 1024
    Wh = synth.weight_rows(4242, N, K)
    X = synth.activations(4243, 2, K)
    Y = q4k.matmul(Wh.to(DEV), N, K, X.to(DEV))
    torch.cuda.synchronize()
    assert q4k.q4k_device_error(clear=False) == 0
    Yr, A = oracle_mod.matmul(Wh.numpy(), N, K, X.numpy())
    assert np.max(np.abs(Y.cpu().double().numpy() - Yr) / (1e-4 * A + 1e-30)) <= 1.0


def test_timeout_on_a_side_stream(q4k):
    s = torch.cuda.Stream()
    q4k.q4k_selftest_timeout(10_000, stream=s)
    s.synchronize()
    assert q4k.q4k_device_error(clear=True) == q4k.Q4K_ERR_TIMEOUT
