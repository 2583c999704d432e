"""Failure detection on the GPU without a fault: a bounded in-kernel wait that can never
complete (an mbarrier nothing arrives on) gives up after its limit, the device status word
reports ATTN_ERR_DEVICE_TIMEOUT to the host, the word is cleared by reading it, and the
context keeps working for the next call.  The timeout is also visible without a
synchronisation (attn_last_device_status), and the next launching call refuses with it."""
import time

import pytest
import torch

from attn_fwd_02_gb300 import workloads

pytestmark = pytest.mark.gpu
DEVICE_TIMEOUT = 6


def test_bounded_wait_reports_timeout_and_context_survives(oracle_mod):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attn_fwd_02_gb300 import binding, build
    build.build()
    assert binding.attn_check_device_status() == 0  # clean before
    assert binding.attn_last_device_status() == 0
    t0 = time.time()
    binding.attn_selftest_bounded_wait()
    assert binding.attn_check_device_status() == DEVICE_TIMEOUT
    elapsed = time.time() - t0
    assert 1.0 < elapsed < 30.0, elapsed  # the wait ran for about its two-second limit
    assert binding.attn_check_device_status() == 0  # reading clears it
    assert binding.attn_last_device_status() == 0
    # the context is still usable: a normal prefill call matches the oracle
    shape = workloads.PrefillShape("after timeout", 1, 2, 200, 200, 64, True, seed=60)
    inp = workloads.prefill_inputs(shape)
    o, lse = binding.attn_fwd(inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda(), True, shape.scale)
    torch.cuda.synchronize()
    assert binding.attn_check_device_status() == 0
    o_ref, lse_ref = oracle_mod.attn_fwd(inp["q"], inp["k"], inp["v"], True, shape.scale)
    assert abs(o.float().cpu().numpy() - o_ref).max() <= 1e-2
    assert abs(lse.cpu().numpy() - lse_ref).max() <= 1e-3


def test_timeout_is_reported_on_the_next_call_without_a_sync(oracle_mod):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attn_fwd_02_gb300 import binding, build
    build.build()
    assert binding.attn_check_device_status() == 0
    shape = workloads.PrefillShape("after timeout", 1, 2, 200, 200, 64, True, seed=61)
    inp = workloads.prefill_inputs(shape)
    q, k, v = inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda()
    binding.attn_selftest_bounded_wait()
    # the host-visible flag is set by the kernel itself once its wait gives up; poll it
    # with plain reads (no stream synchronisation), for at most 30 s
    t0 = time.time()
    while binding.attn_last_device_status() == 0 and time.time() - t0 < 30.0:
        time.sleep(0.05)
    assert binding.attn_last_device_status() == DEVICE_TIMEOUT
    assert binding.attn_last_device_status() == DEVICE_TIMEOUT  # reading does not clear it
    # the next launching call refuses, launches nothing and leaves its outputs alone
    o = torch.full_like(q, 7.0)
    with pytest.raises(binding.AttnError) as ei:
        binding.attn_fwd(q, k, v, True, shape.scale, out=o)
    assert ei.value.status == DEVICE_TIMEOUT
    torch.cuda.synchronize()
    assert bool((o == 7.0).all())
    # the synchronising check reports and clears; calls work again
    assert binding.attn_check_device_status() == DEVICE_TIMEOUT
    assert binding.attn_last_device_status() == 0
    o, lse = binding.attn_fwd(q, k, v, True, shape.scale)
    torch.cuda.synchronize()
    assert binding.attn_check_device_status() == 0
    o_ref, lse_ref = oracle_mod.attn_fwd(inp["q"], inp["k"], inp["v"], True, shape.scale)
    assert abs(o.float().cpu().numpy() - o_ref).max() <= 1e-2
    assert abs(lse.cpu().numpy() - lse_ref).max() <= 1e-3
