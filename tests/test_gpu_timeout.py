"""The failure path of the library's bounded waits, exercised without faulting the GPU: a wait
on an mbarrier phase that nothing completes gives up after its limit, the device error word
reports KDA_ERR_TIMEOUT once (and is cleared by reading it), and the context stays usable."""

import pytest
import torch

from kimi_delta_attention_02_gb300 import binding, workloads

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_reports():
    binding.check_device_error()  # nothing pending from earlier work
    assert binding.selftest_wait_timeout() == 1
    with pytest.raises(binding.KdaError) as e:
        binding.check_device_error()
    assert e.value.status == binding.KDA_ERR_TIMEOUT
    binding.check_device_error()  # cleared by the read
    # the context still runs kernels
    case = workloads.make_prefill([40], H=2, device="cuda", seed=60)
    out, fin = binding.prefill(case.q, case.k, case.v, case.log_alpha, case.beta, case.cu_seqlens,
                               case.init_state)
    binding.check_device_error()
    assert torch.isfinite(out).all() and torch.isfinite(fin).all()
