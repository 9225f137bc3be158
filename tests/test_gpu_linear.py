"""Parity of mla_linear (through the C ABI) with the oracle's y = x W^T.

bf16 inputs, fp32 accumulation, bf16 output: every element within half a bf16
step of the fp64 result plus the accumulation error of K terms in fp32
(|err| <= 2^-9 |y| + K 2^-23 sum_k |x_k w_k|), with shapes that cover partial
output tiles, K splits (with and without) and token counts from 1 to 256.
"""

import numpy as np
import pytest
import torch

from oracle import mla_oracle as O

pytestmark = pytest.mark.gpu


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("T,K,N", [(1, 64, 1), (32, 7168, 512), (32, 7168, 64), (32, 1536, 16384),
                                   (7, 16384, 7168), (256, 512, 300), (100, 1536, 8192), (32, 7168, 1536)])
def test_linear_parity(T, K, N):
    from mla_absorbed_decode_absorb_gb300 import ops
    g = torch.Generator().manual_seed(T * 131 + K + N)
    x = torch.randn(T, K, generator=g).to(torch.bfloat16)
    w = (torch.randn(N, K, generator=g) / K ** 0.5).to(torch.bfloat16)
    y = ops.mla_linear(x.cuda(), w.cuda())
    torch.cuda.synchronize()
    assert ops.mla_get_device_status() == ops.MLA_OK
    xf, wf = O.bf16_bits_to_f64(bits(x)), O.bf16_bits_to_f64(bits(w))
    ref = O.linear(xf, wf)
    mag = np.abs(xf) @ np.abs(wf).T
    got = y.float().cpu().numpy()
    tol = 2.0 ** -8 * np.abs(ref) + K * 2.0 ** -23 * mag + 1e-30
    assert (np.abs(got - ref) <= tol).all(), np.abs(got - ref).max()


@pytest.mark.parametrize("T,K,N0,N1", [(32, 7168, 512, 64), (1, 64, 1, 130), (100, 1536, 300, 8192)])
def test_linear_pair_parity(T, K, N0, N1):
    """Two projections of one x in one launch, each against the oracle's x W^T."""
    from mla_absorbed_decode_absorb_gb300 import ops
    g = torch.Generator().manual_seed(T * 7 + K + N0 + 3 * N1)
    x = torch.randn(T, K, generator=g).to(torch.bfloat16)
    w0 = (torch.randn(N0, K, generator=g) / K ** 0.5).to(torch.bfloat16)
    w1 = (torch.randn(N1, K, generator=g) / K ** 0.5).to(torch.bfloat16)
    y0, y1 = ops.mla_linear_pair(x.cuda(), w0.cuda(), w1.cuda())
    torch.cuda.synchronize()
    assert ops.mla_get_device_status() == ops.MLA_OK
    xf = O.bf16_bits_to_f64(bits(x))
    for w, y in ((w0, y0), (w1, y1)):
        wf = O.bf16_bits_to_f64(bits(w))
        ref = O.linear(xf, wf)
        mag = np.abs(xf) @ np.abs(wf).T
        tol = 2.0 ** -8 * np.abs(ref) + K * 2.0 ** -23 * mag + 1e-30
        assert (np.abs(y.float().cpu().numpy() - ref) <= tol).all()


def test_linear_rejects_bad_shapes():
    from mla_absorbed_decode_absorb_gb300 import ops
    x = torch.zeros(4, 96, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(8, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ops.MLAError):
        ops.mla_linear(x, w)        # K not a multiple of 64
    x = torch.zeros(257, 64, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(8, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ops.MLAError):
        ops.mla_linear(x, w)        # T > 256
