"""The bounded-wait path, exercised without faulting the GPU: a diagnostic kernel waits on a barrier
nothing arrives on, gives up after a short limit and records the timeout in the device status word;
the host reads it as ATTNFUSE_ERR_TIMEOUT and the context stays usable."""
import math

import pytest
import torch

from attention_rope_causal_gb300 import binding, build, inputs

pytestmark = pytest.mark.gpu

TIMEOUT = 4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load()


def test_wait_timeout_is_reported_and_cleared():
    assert binding.device_status() == 0
    binding.diag_wait_timeout(10_000_000)  # 10 ms
    assert binding.device_status() == TIMEOUT
    assert "ran out" in binding.last_error()
    assert binding.device_status() == 0  # reading clears it


def test_kernels_stand_down_while_a_timeout_is_unread_then_recover():
    w = inputs.TINY
    q, k, v = (t.cuda() for t in inputs.make_inputs(w))
    good, _ = binding.rope_causal_fwd(q, k, v, w.rope_base)
    torch.cuda.synchronize()
    binding.diag_wait_timeout(5_000_000)
    out = torch.full_like(q, math.nan)
    binding.rope_causal_fwd(q, k, v, w.rope_base, out=out)
    assert binding.device_status() == TIMEOUT
    assert torch.isnan(out.float()).all()  # the attention kernel did no work
    out2, _ = binding.rope_causal_fwd(q, k, v, w.rope_base)
    assert binding.device_status() == 0
    assert torch.equal(out2, good)
