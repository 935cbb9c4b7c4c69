"""The pipe-rate probes behind the benchmark's rooflines: each launch performs
the operation count it reports (threads x steps x counted operations per
step), the count scales with the steps, the launch time grows with the
steps (no chain folded away), and the rates come out in the order the
hardware's unit counts put them (the transcendental pipe slowest, the fp32
pipe's FLOP rate highest), none above the instruction issue limit."""
import pytest

import token_perturbation_estimator_gb300 as dust
from helpers import cuda

pytestmark = pytest.mark.gpu

OPS_PER_THREAD_STEP = {dust.PIPE_XU: 32, dust.PIPE_ALU: 24, dust.PIPE_FMA: 16,
                       dust.PIPE_ISSUE: 32}


def _rate(pipe, steps, sink):
    import torch
    s = torch.cuda.current_stream()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    dust.dust_pipe_probe(pipe, steps, sink, s)  # warm
    a.record(s)
    ops = dust.dust_pipe_probe(pipe, steps, sink, s)
    b.record(s)
    b.synchronize()
    return ops, ops / (a.elapsed_time(b) * 1e-3)


def test_probe_counts_and_rate_order():
    import torch
    dev = cuda()
    n = dust.dust_pipe_probe_threads()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    assert n == sms * 4 * 512
    sink = torch.zeros(n, dtype=torch.float32, device=dev)
    rates = {}
    for pipe, per in OPS_PER_THREAD_STEP.items():
        ops, rate = _rate(pipe, 2048, sink)
        assert ops == n * 2048 * per
        ops4, rate4 = _rate(pipe, 8192, sink)
        assert ops4 == 4 * ops
        # four times the steps take well over twice the time
        assert rate4 < 2 * rate
        rates[pipe] = rate4
    torch.cuda.synchronize()
    assert dust.dust_last_error() == dust.OK
    assert 0 < rates[dust.PIPE_XU] < rates[dust.PIPE_ALU] < rates[dust.PIPE_FMA]
    assert rates[dust.PIPE_XU] < rates[dust.PIPE_ISSUE]
    # No probe may beat the instruction issue limit of 4 warp instructions
    # per clock per SM (ALU and issue count lane instructions, FMA 2 FLOP each)
    # at the highest SM clock this GPU reports.
    khz = getattr(torch.cuda.get_device_properties(dev), "clock_rate", 0)
    mhz = khz / 1000.0 if khz else 2100.0
    limit = 128.0 * sms * mhz * 1e6 * 1.02
    assert rates[dust.PIPE_ALU] < limit and rates[dust.PIPE_ISSUE] < limit
    assert rates[dust.PIPE_FMA] < 2 * limit
