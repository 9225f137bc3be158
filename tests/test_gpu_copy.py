"""mla_copy_async: the step's transport between pinned host memory and the device.

Byte-exact copies device->device, pinned host->device and device->pinned host,
at sizes around the 16-byte vector width, at misaligned offsets and at the
size of a decode step's inputs; refusals of pageable host memory and of
overlapping ranges; and a decode step run end to end through the session's
upload / download equal to the device-resident step.
"""

import numpy as np
import pytest
import torch

from mla_absorbed_decode_absorb_gb300 import workloads as W

pytestmark = pytest.mark.gpu

SIZES = [1, 15, 16, 17, 4099, 65536 + 7, 1610240]


def _rand(n, seed):
    g = np.random.default_rng(seed)
    return torch.from_numpy(g.integers(0, 256, size=n, dtype=np.uint8))


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("offset", [0, 3])
def test_copy_device_and_host(n, offset):
    from mla_absorbed_decode_absorb_gb300 import ops
    src_h = _rand(n + offset, n).pin_memory()
    dev = torch.zeros(n + 2 * offset, dtype=torch.uint8, device="cuda")
    ops.mla_copy(dev[offset:offset + n], src_h[offset:])                # host -> device
    back = torch.zeros(n + offset, dtype=torch.uint8).pin_memory()
    dev2 = torch.zeros(n, dtype=torch.uint8, device="cuda")
    ops.mla_copy(dev2, dev[offset:offset + n])                         # device -> device
    ops.mla_copy(back[offset:], dev2)                                  # device -> host
    torch.cuda.synchronize()
    assert torch.equal(back[offset:], src_h[offset:])
    assert torch.equal(dev[offset:offset + n].cpu(), src_h[offset:])
    assert ops.mla_get_device_status() == ops.MLA_OK


def test_out_projection_refuses_pageable_output():
    from mla_absorbed_decode_absorb_gb300 import ops
    o = torch.zeros(1, 1, 128, 512, dtype=torch.float32, device="cuda")
    w = torch.zeros(128, 128, 512, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        ops.mla_out_absorb(o, w, torch.zeros(1, 1, 128, 128, dtype=torch.bfloat16))
    pageable = torch.zeros(1, 1, 128, 128, dtype=torch.bfloat16)
    assert ops.lib.mla_out_absorb(o.data_ptr(), w.data_ptr(), pageable.data_ptr(), 1, 1, 0) == ops.MLA_ERR_INVALID_ARG


def test_copy_refusals():
    from mla_absorbed_decode_absorb_gb300 import ops
    dev = torch.zeros(256, dtype=torch.uint8, device="cuda")
    pageable = torch.zeros(256, dtype=torch.uint8)
    with pytest.raises(ValueError):
        ops.mla_copy(dev, pageable)
    # the C entry point refuses pageable memory and overlapping ranges by itself
    assert ops.lib.mla_copy_async(dev.data_ptr(), pageable.data_ptr(), 256, 0) == ops.MLA_ERR_INVALID_ARG
    assert ops.lib.mla_copy_async(dev.data_ptr() + 16, dev.data_ptr(), 64, 0) == ops.MLA_ERR_INVALID_ARG
    assert ops.lib.mla_copy_async(dev.data_ptr(), dev.data_ptr(), 0, 0) == ops.MLA_OK
    with pytest.raises(ValueError):
        ops.mla_copy(dev[:128], dev[128:].clone()[:64])


@pytest.mark.parametrize("level", [1, 2])
def test_step_through_host_buffers(level):
    """upload -> step -> download gives the device-resident step's output, bit for bit."""
    from mla_absorbed_decode_absorb_gb300 import ops
    from mla_absorbed_decode_absorb_gb300.runtime import DecodeSession
    before = ops.mla_get_launch_overlap()
    ops.mla_set_launch_overlap(level)
    try:
        inp = W.generate(W.custom("host_io", [5, 700, 64], n_q=2), seed=13)
        ref = DecodeSession(inp)
        ref.step()
        s = DecodeSession(inp)
        host_in = s.host_step_buffer(pin=True)
        s.step_buffer.zero_()                       # the inputs now come only from the host
        host_out = torch.empty(s.out.shape, dtype=s.out.dtype).pin_memory()
        for _ in range(2):
            s.upload(host_in)
            s.step()
            s.download(host_out)
        torch.cuda.synchronize()
        assert ops.mla_get_device_status() == ops.MLA_OK
        assert torch.equal(host_out.view(torch.int16), ref.out.cpu().view(torch.int16))
        # the out-projection storing straight into the pinned buffer
        host_out.zero_()
        for fused in (True, False):
            t = DecodeSession(inp, fused_finish=fused)
            t.step_buffer.zero_()
            t.upload(host_in)
            assert t.step(host_out=host_out) is host_out
            torch.cuda.synchronize()
            assert ops.mla_get_device_status() == ops.MLA_OK
            assert torch.equal(host_out.view(torch.int16), ref.out.cpu().view(torch.int16))
            host_out.zero_()
    finally:
        ops.mla_set_launch_overlap(before)
