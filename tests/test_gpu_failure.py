"""Failure detection on the GPU without a fault: a pipeline wait that runs out raises the
timeout bit of the device status word and returns, and the context stays usable."""
import pytest
import torch

from paged_kv_chunk_gb300 import capi
from paged_kv_chunk_gb300 import synthetic as syn

from helpers import check_close, gpu_stream_inputs, oracle_chunk, stream_case, to_np

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_the_context_stays_usable():
    capi.oasr_device_status(clear=True)
    capi.oasr_selftest_wait(20000)          # a barrier nothing signals, 20 ms limit
    assert capi.oasr_device_status(clear=True) == capi.STATUS_TIMEOUT_BIT
    # the next launches run normally and raise nothing
    cfg = syn.TINY
    x = stream_case(cfg)
    d = gpu_stream_inputs(x, cfg.dtype)
    out = capi.oasr_chunk_step_paged(d["q"], d["k_new"], d["v_new"], d["k_pool"], d["v_pool"],
                                     d["block_table"], d["cache_seqlens"], d["pos_bias_u"],
                                     d["pos_bias_v"], d["rel"])
    torch.cuda.synchronize()
    check_close(to_np(out), oracle_chunk(x), cfg.dtype, "after a timed-out wait")
    assert capi.oasr_device_status() == 0


def test_timeout_bit_is_cleared_on_read():
    capi.oasr_selftest_wait(1000)
    assert capi.oasr_device_status(clear=False) == capi.STATUS_TIMEOUT_BIT
    assert capi.oasr_device_status(clear=True) == capi.STATUS_TIMEOUT_BIT
    assert capi.oasr_device_status() == 0
